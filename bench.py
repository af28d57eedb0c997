#!/usr/bin/env python
"""Benchmark of the fp8 e4m3 KV cache hot path on one GB300 (or N replicas).

One step = one decode step of the 64-sequence full-attention workload
(64 seqs, 32 q / 4 KV heads, head_dim 128, contexts U[1K, 32K], block 16,
bf16 relative bias of extent 1,024), made by paged_attn_fp8_decode_store in
two launches:
  the running amax over the step's new K/V tokens  (calibration pass)
  the store of the new tokens into the cache        (quant-on-store)
  fp8 attention over the whole cache + split merge  (fp8 attention)
`value` is the step's algorithmic HBM bytes / step time (GB/s); the same step
as separate calls (kv_amax_calibrate, kv_store_e4m3, paged_attn_fp8_decode)
is timed beside it under "separate_calls".  The other
workloads (varlen prefill, 128K calibrated decode, 1M decode) are measured the
same way and reported under "extra".

--impl reference times the CPU oracle (float64, plain C) on a bounded sample
of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "fp8-KV decode attn HBM GB/s (% of ~8 TB/s); prefill fp8 TFLOP/s"


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            m = json.load(f)
        return {"hbm_gbs": float(m["hbm_gbs"]), "bf16_tflops": float(m["bf16_tflops"]),
                "bf16_tflops_sustained": float(m.get("bf16_tflops_sustained", m["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def fp8_mma_probe(dev, shapes=((256, 2, 1), (128, 2, 2), (128, 1, 1), (64, 2, 2))):
    """FP8 (e4m3) tcgen05 MMA throughput of this GPU measured by the repo's
    own probe (libfp8kv_probe.so): one CTA per SM, `issuers` threads issuing
    M=128, K=32 MMAs of N = n back to back over `accs` accumulators each,
    timed with CUDA events.  Context for the prefill roofline, whose
    denominator stays 2 x the measured bf16 rate."""
    import ctypes
    path = os.path.join(ROOT, "fp8_e4m3_kv_gb300", "libfp8kv_probe.so")
    if not os.path.exists(path):
        return None
    lib = ctypes.CDLL(path)
    fn = lib.fp8kv_probe_mma_e4m3_mode
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                   ctypes.c_int32, ctypes.POINTER(ctypes.c_float), ctypes.c_void_p]
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    res = {}
    for shape in shapes:
        n, accs, issuers = shape[:3]
        mode = shape[3] if len(shape) > 3 else 0
        iters = 20000 * 256 // n
        ms = ctypes.c_float()
        rc = fn(sms, iters, n, accs, issuers, mode, ctypes.byref(ms),
                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        if rc != 0 or ms.value <= 0:
            return {"error": "probe status %d" % rc}
        key = "n%d_acc%d_thr%d" % (n, accs, issuers) + ("_mode%d" % mode if mode else "")
        res[key + "_tflops"] = 2.0 * 128 * n * 32 * iters * issuers * sms / (ms.value * 1e-3) / 1e12
    return res


# DRAM bytes (read + write) of one decode launch of the 64-sequence workload,
# from the ncu capture summarised in profiles/ (decode launch list: measured
# on a 16-sequence cut and scaled by the KV bytes), keyed by a hash of the
# kernel sources it was taken on: once the kernel changes, the number no
# longer describes it and is reported as null.
DECODE_TRAFFIC = {
    "5843f6d234db49262a04ebf0e60c29ce4789645d24dfbab2cb22e29c499e6c3b": 1086198746,
}
DECODE_SOURCES = ("fp8_e4m3_kv_gb300/csrc/attn_decode.cu", "fp8_e4m3_kv_gb300/csrc/common.cuh")


def decode_sources_sha():
    import hashlib
    h = hashlib.sha256()
    for rel in DECODE_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def decode_traffic_bytes():
    return DECODE_TRAFFIC.get(decode_sources_sha())


# ---------------------------------------------------------------------------
# distributed plumbing (replicas only: no data-path collective)
# ---------------------------------------------------------------------------
def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world <= 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# workloads on the device
# ---------------------------------------------------------------------------
class DecodeRun:
    """A decode workload resident in HBM: cache filled once, then each step
    calibrates + stores the step's new token per sequence and decodes."""

    def __init__(self, fk, spec, dev, seed=0, scales=(1.0, 1.0, 1.0), calibrate=False):
        self.fk, self.spec, self.dev = fk, spec, dev
        inp = workloads.make_decode(spec, device=dev, seed=seed)
        kv = inp["kv"]
        self.inp, self.kv = inp, kv
        sq, sk, sv = scales
        self.amax = torch.zeros(3, dtype=torch.float32, device=dev)
        if calibrate:
            fk.kv_amax_calibrate(kv.k, kv.v, self.amax[0:1], self.amax[1:2], kv.slot_mapping)
            fk.kv_amax_calibrate(inp["q"], None, self.amax[2:3], None)
            ak, av, aq = self.amax.cpu().tolist()
            sk, sv, sq = fk.scale_from_amax(ak), fk.scale_from_amax(av), fk.scale_from_amax(aq)
        self.scales = (sq, sk, sv)
        self.cache = fk.KVCache.empty(kv.num_blocks, kv.block_size, spec.Hkv, spec.D, device=dev)
        fk.kv_store_e4m3(self.cache, kv.k, kv.v, kv.slot_mapping, sk, sv)
        # the step's new token of each sequence is its last one
        lens = inp["lens"]
        last = torch.tensor([s + L - 1 for s, L in zip(kv.tok_start.tolist()[:-1], lens)],
                            dtype=torch.int64, device=dev)
        self.k_new = kv.k[last].contiguous()
        self.v_new = kv.v[last].contiguous()
        self.slot_new = kv.slot_mapping[last].contiguous()
        self.q = inp["q"]
        self.rel = inp["rel"]
        self.out = torch.empty_like(self.q)
        B, Hq, D = self.q.shape
        n = fk.decode_workspace_size(B, Hq, spec.Hkv, D, kv.max_blocks, kv.block_size,
                                     spec.window, 0)
        self.ws = torch.empty(n, dtype=torch.uint8, device=dev)
        self.step_amax = torch.zeros(2, dtype=torch.float32, device=dev)
        self.amax_views = (self.step_amax[0:1], self.step_amax[1:2])
        torch.cuda.synchronize()
        # algorithmic bytes
        E = 0 if self.rel is None else self.rel.shape[2]
        kv_bytes = sum(min(L, spec.window) if spec.window else L for L in lens) * spec.Hkv * D * 2
        self.decode_bytes = kv_bytes + 2 * B * Hq * D * 2 + B * Hq * E * 2
        nt = B * spec.Hkv * D
        self.store_bytes = nt * 2 * (2 + 1)     # read bf16 K and V, write e4m3 K and V
        self.amax_bytes = nt * 2 * 2
        self.step_bytes = self.decode_bytes + self.store_bytes + self.amax_bytes
        self.launches_per_step = 2              # fused store + amax + decode, merge
        # the same decode bound to these buffers (validated once, no per-call
        # checks): the host's part of a call is then the C entry point alone
        self.bound = fk.DecodeStep(self.cache, self.q, kv.block_table, kv.seq_lens, sq, sk, sv,
                                   rel_bias=self.rel, window=spec.window, out=self.out,
                                   workspace=self.ws)

    def step(self, q=None, k_new=None, v_new=None, seq_lens=None, out=None):
        """One decode step in one call: store each sequence's new token, raise
        the running amax over it, attend."""
        fk, kv = self.fk, self.kv
        sq, sk, sv = self.scales
        return fk.paged_attn_fp8_decode_store(
            self.cache, self.q if q is None else q, self.k_new if k_new is None else k_new,
            self.v_new if v_new is None else v_new, kv.block_table,
            kv.seq_lens if seq_lens is None else seq_lens, sq, sk, sv, rel_bias=self.rel,
            window=self.spec.window, amax_k=self.amax_views[0], amax_v=self.amax_views[1],
            out=self.out if out is None else out, workspace=self.ws)

    def step_separate(self):
        """The same step as three calls (amax, store, decode): four launches."""
        fk = self.fk
        sq, sk, sv = self.scales
        fk.kv_amax_calibrate(self.k_new, self.v_new, self.step_amax[0:1], self.step_amax[1:2],
                             self.slot_new)
        fk.kv_store_e4m3(self.cache, self.k_new, self.v_new, self.slot_new, sk, sv)
        return self.decode()

    def decode(self, q=None, seq_lens=None, out=None):
        sq, sk, sv = self.scales
        return self.fk.paged_attn_fp8_decode(
            self.cache, self.q if q is None else q, self.kv.block_table,
            self.kv.seq_lens if seq_lens is None else seq_lens, sq, sk, sv,
            rel_bias=self.rel, window=self.spec.window, out=self.out if out is None else out,
            workspace=self.ws)


def time_steps(fn, steps, warmup, world):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(steps):
        fn()
    e1.record(s)
    torch.cuda.synchronize()
    barrier(world)
    ms = e0.elapsed_time(e1) / steps
    return max_over_ranks(ms, world)


def e2e_decode(run, steps, warmup, world):
    """Same step through the public API from pinned host memory: per step, one
    copy of the step's inputs (q, new K, new V, lengths, packed in one pinned
    staging buffer at 256-byte offsets) to the device, the call (a DecodeStep
    bound to the staging buffers' device copies, as a decode loop keeps them),
    a read back of out and a host sync.  Timed twice: issued one by one
    ("eager"), and as one CUDA graph of the three (DecodeStep.cuda_graph);
    returns ms per step of each, and the bytes copied each way."""
    parts = {"q": run.q, "k_new": run.k_new, "v_new": run.v_new, "seq_lens": run.kv.seq_lens}
    offs, total = {}, 0
    for k, t in parts.items():
        offs[k] = total
        total += -(-t.numel() * t.element_size() // 256) * 256
    host = torch.empty(total, dtype=torch.uint8).pin_memory()
    dev_buf = torch.empty(total, dtype=torch.uint8, device=run.dev)
    dev = {}
    for k, t in parts.items():
        n = t.numel() * t.element_size()
        host[offs[k]:offs[k] + n].copy_(t.detach().cpu().contiguous().view(-1).view(torch.uint8))
        dev[k] = dev_buf[offs[k]:offs[k] + n].view(t.dtype).view(t.shape)
    out_h = torch.empty(run.out.shape, dtype=run.out.dtype).pin_memory()
    h2d = total
    d2h = out_h.numel() * out_h.element_size()
    sq, sk, sv = run.scales
    step = run.fk.DecodeStep(run.cache, dev["q"], run.kv.block_table, dev["seq_lens"], sq, sk, sv,
                             rel_bias=run.rel, window=run.spec.window, out=run.out,
                             workspace=run.ws, k_new=dev["k_new"], v_new=dev["v_new"],
                             amax_k=run.amax_views[0], amax_v=run.amax_views[1])

    def copy_in():
        dev_buf.copy_(host, non_blocking=True)

    def copy_out():
        out_h.copy_(run.out, non_blocking=True)

    def eager():
        copy_in()
        step.run()
        copy_out()
    # the same step as one CUDA graph (copy in, store + decode, read back)
    graph = step.cuda_graph(pre=copy_in, post=copy_out)
    res = {}
    for name, one in (("eager", eager), ("graph", graph.replay)):
        for _ in range(warmup):
            one()
        torch.cuda.synchronize()
        barrier(world)
        t0 = time.perf_counter()
        for _ in range(steps):
            one()
            torch.cuda.current_stream().synchronize()   # the result is on the host each step
        ms = (time.perf_counter() - t0) * 1e3 / steps
        res[name] = max_over_ranks(ms, world)
    return res, h2d, d2h


# ---------------------------------------------------------------------------
# CPU oracle baseline (bounded sample)
# ---------------------------------------------------------------------------
def oracle_decode_sample(spec, inp, scales, budget_s=15.0, max_keys=None):
    """Time the oracle on whole sequences of the workload (all heads), one
    after another, until about budget_s of CPU work; returns GB/s over the
    sample's KV bytes and a description.  With max_keys, a longer sequence is
    cut to its first max_keys keys (a decode of that shorter sequence: same
    heads, bias and window, the query at its last kept key); the oracle's
    cost is linear in the keys, so GB/s carries over to the full lengths."""
    import oracle
    bits = workloads.bf16_bits
    kv = inp["kv"]
    sq, sk, sv = scales
    q = inp["q"]
    B, Hq, D = q.shape
    G = Hq // spec.Hkv
    lens = inp["lens"]
    starts = kv.tok_start.cpu().tolist()
    done_bytes, t_total, seqs = 0, 0.0, 0
    for b in range(B):
        L = lens[b] if max_keys is None else min(lens[b], max_keys)
        L_used = min(L, spec.window) if spec.window else L
        kb = bits(kv.k[starts[b]:starts[b] + L])
        vb = bits(kv.v[starts[b]:starts[b] + L])
        qb = bits(q[b])
        relb = None if inp["rel"] is None else bits(inp["rel"][b])
        t0 = time.perf_counter()
        k8 = oracle.quantize(kb, sk)
        v8 = oracle.quantize(vb, sv)
        q8 = oracle.quantize(qb, sq)
        rows = Hq
        q_off = np.arange(rows, dtype=np.int64) * D
        kv_off = (np.arange(rows) // G) * D
        bias_off = None if relb is None else np.arange(rows, dtype=np.int64) * relb.shape[-1]
        oracle.attend_rows(D, q8, q_off, k8, v8, kv_off, spec.Hkv * D, [L] * rows,
                           [L - 1] * rows, 1 / math.sqrt(D), sq, sk, sv, relb, bias_off,
                           0 if relb is None else relb.shape[-1], spec.window)
        t_total += time.perf_counter() - t0
        done_bytes += L_used * spec.Hkv * D * 2
        seqs += 1
        if t_total >= budget_s:
            break
    return done_bytes / t_total / 1e9, seqs, t_total, oracle.num_threads()


def cpu_line(value, unit, cores, sample):
    return {"value": value, "unit": unit, "cores": cores, "kind": "oracle", "sample": sample}


def oracle_decode_baseline(spec, inp, scales, budget_s, max_keys=None):
    gbs, seqs, t, cores = oracle_decode_sample(spec, inp, scales, budget_s, max_keys)
    cut = "" if max_keys is None else ", each cut to its first %d keys" % max_keys
    return cpu_line(gbs, "GB/s", cores, "%d sequence(s) of the workload (all %d q heads, float64)%s,"
                    " %.1f s of CPU time; GB/s over the sample's KV bytes" % (seqs, spec.Hq, cut, t))


def oracle_prefill_baseline(spec, inp, groups, budget_s, seed=0):
    """The oracle on the prefill chunk: the quantization of every sequence's K
    and V (timed in full), then query rows drawn from every sequence and head
    (each quantized and attended over all its visible keys) until about
    budget_s of CPU time.  The time of the whole chunk is extrapolated as
    quantization + (row time) x (all rows / rows done); TFLOP/s is the
    chunk's visible-pair FLOPs over that time."""
    import oracle
    bits = workloads.bf16_bits
    kv = inp["kv"]
    D, Hq, Hkv = spec.D, spec.Hq, spec.Hkv
    G = Hq // Hkv
    rng = np.random.default_rng(seed)
    cu = inp["cu_seqlens_q"].tolist()
    starts = kv.tok_start.cpu().tolist()
    t_quant, codes = 0.0, {}
    for b, _ in groups:
        kn = inp["k_lens"][b]
        kb = bits(kv.k[starts[b]:starts[b] + kn])
        vb = bits(kv.v[starts[b]:starts[b] + kn])
        t0 = time.perf_counter()
        codes[b] = (oracle.quantize(kb, 1.0), oracle.quantize(vb, 1.0))
        t_quant += time.perf_counter() - t0
    t_rows, rows_done, rows_all, flops_all = 0.0, 0, 0, 0
    for b, w in groups:
        qn, kn = inp["q_lens"][b], inp["k_lens"][b]
        rows_all += qn * Hq
        flops_all += Hq * sum(4 * D * (min(kn - qn + i + 1, w) if w else kn - qn + i + 1)
                              for i in range(qn))
    while t_rows < budget_s:
        for b, w in groups:
            qn, kn = inp["q_lens"][b], inp["k_lens"][b]
            ts = rng.integers(0, qn, 8)
            hs = rng.integers(0, Hq, 8)
            qb = np.stack([bits(inp["q"][cu[b] + int(t), int(h)]) for t, h in zip(ts, hs)])
            relb = None if inp["rel"] is None else np.stack(
                [bits(inp["rel"][cu[b] + int(t), int(h)]) for t, h in zip(ts, hs)])
            E = 0 if relb is None else relb.shape[-1]
            n = len(ts)
            k8, v8 = codes[b]
            t0 = time.perf_counter()
            q8 = oracle.quantize(qb, 1.0)
            oracle.attend_rows(D, q8, np.arange(n, dtype=np.int64) * D, k8, v8,
                               (hs // G).astype(np.int64) * D, Hkv * D, [kn] * n,
                               [kn - qn + int(t) for t in ts], 1 / math.sqrt(D), 1.0, 1.0, 1.0,
                               relb, None if relb is None else np.arange(n, dtype=np.int64) * E,
                               E, w)
            t_rows += time.perf_counter() - t0
            rows_done += n
    t_est = t_quant + t_rows * rows_all / rows_done
    return cpu_line(flops_all / t_est / 1e12, "TFLOP/s", oracle.num_threads(),
                    "K/V quantization of every sequence (%.1f s) plus %d of the chunk's %d query "
                    "rows drawn from every sequence and head (%.1f s, float64, each over all its "
                    "visible keys); whole-chunk time extrapolated linearly in rows: %.0f s"
                    % (t_quant, rows_done, rows_all, t_rows, t_est))


# ---------------------------------------------------------------------------
# secondary workloads
# ---------------------------------------------------------------------------
def bench_prefill(fk, dev, steps, warmup, world, only_group=None, cpu_budget=0.0):
    spec = workloads.PREFILL_16K
    inp = workloads.make_prefill(spec, device=dev, seed=0)
    kv = inp["kv"]
    cache = fk.KVCache.empty(kv.num_blocks, kv.block_size, spec.Hkv, spec.D, device=dev)
    q_lens = inp["q_lens"]
    half = spec.n_seqs // 2
    groups = []
    cu = inp["cu_seqlens_q"].tolist()
    for gi, (lo, hi) in enumerate([(0, half), (half, spec.n_seqs)]):
        w = spec.windows[gi]
        cu_g = torch.tensor([c - cu[lo] for c in cu[lo:hi + 1]], dtype=torch.int32, device=dev)
        groups.append(dict(window=w, q=inp["q"][cu[lo]:cu[hi]], cu=cu_g,
                           lens=kv.seq_lens[lo:hi].contiguous(),
                           bt=kv.block_table[lo:hi].contiguous(),
                           rel=inp["rel"][cu[lo]:cu[hi]],
                           out=torch.empty_like(inp["q"][cu[lo]:cu[hi]]),
                           maxq=max(q_lens[lo:hi])))
    flops = 0
    for gi, (lo, hi) in enumerate([(0, half), (half, spec.n_seqs)]):
        if only_group is not None and gi != only_group:
            continue
        w = spec.windows[gi]
        for L in q_lens[lo:hi]:
            flops += sum(min(i + 1, w) if w else i + 1 for i in range(L))
    flops *= 4 * spec.Hq * spec.D
    if only_group is not None:
        fk.kv_store_e4m3(cache, kv.k, kv.v, kv.slot_mapping, 1.0, 1.0)
        groups = [groups[only_group]]

    def step():
        if only_group is None:
            fk.kv_store_e4m3(cache, kv.k, kv.v, kv.slot_mapping, 1.0, 1.0)
        for g in groups:
            fk.attn_fp8_varlen_prefill(cache, g["q"], g["cu"], g["lens"], g["bt"], g["maxq"],
                                       1.0, 1.0, 1.0, rel_bias=g["rel"], window=g["window"],
                                       out=g["out"])
    try:
        step()
    except Exception as e:  # noqa: BLE001
        return {"workload": spec.name, "unavailable": str(e)}
    ms = time_steps(step, steps, warmup, world)
    # each group alone (causal, 512-window), the store of the chunk included
    # in neither
    per_group = []
    if only_group is None:
        fk.kv_store_e4m3(cache, kv.k, kv.v, kv.slot_mapping, 1.0, 1.0)
        for gi, (lo, hi) in enumerate([(0, half), (half, spec.n_seqs)]):
            w = spec.windows[gi]
            g = groups[gi]
            gf = 4 * spec.Hq * spec.D * sum(
                sum(min(i + 1, w) if w else i + 1 for i in range(L)) for L in q_lens[lo:hi])

            def one(g=g):
                fk.attn_fp8_varlen_prefill(cache, g["q"], g["cu"], g["lens"], g["bt"], g["maxq"],
                                           1.0, 1.0, 1.0, rel_bias=g["rel"], window=g["window"],
                                           out=g["out"])
            gms = time_steps(one, steps, warmup, world)
            per_group.append({"window": w, "ms": gms, "tflops": gf / gms / 1e9})
    pk = peaks()
    fp8_peak = 2.0 * pk["bf16_tflops"]      # nominal fp8 : bf16 dense ratio of 2
    probe = fp8_mma_probe(dev)
    res = {"workload": spec.name, "ms_per_step": ms, "tflops": flops / ms / 1e9,
           "fp8_mma_probe": probe,
           "roofline": {"bound": "tensor", "achieved": flops / ms / 1e9, "peak": fp8_peak,
                        "unit": "TFLOP/s", "frac": flops / ms / 1e9 / fp8_peak,
                        "peak_source": "2 x %s bf16 burst" % pk["source"]},
           "flops_per_step": flops, "tokens": sum(q_lens),
           "step": "kv_store_e4m3 of the chunk, then one prefill call per group",
           "groups": per_group}
    if cpu_budget > 0:
        res["cpu_baseline"] = oracle_prefill_baseline(
            spec, inp, [(b, spec.windows[0 if b < half else 1]) for b in range(spec.n_seqs)],
            cpu_budget)
    return res


def bench_prefill_per_token(fk, dev, steps, warmup, world):
    """The prefill chunk's two groups (causal, 512-window) over a cache written
    by kv_store_e4m3_per_token; the store is outside the timed calls."""
    spec = workloads.PREFILL_16K
    inp = workloads.make_prefill(spec, device=dev, seed=0)
    kv = inp["kv"]
    cache = fk.KVCache.empty(kv.num_blocks, kv.block_size, spec.Hkv, spec.D, device=dev)
    ks = torch.empty((kv.num_blocks, spec.Hkv, kv.block_size), dtype=torch.float32, device=dev)
    vs = torch.empty_like(ks)
    fk.kv_store_e4m3_per_token(cache, kv.k, kv.v, kv.slot_mapping, ks, vs)
    q_lens = inp["q_lens"]
    half = spec.n_seqs // 2
    cu = inp["cu_seqlens_q"].tolist()
    groups, flops = [], 0
    for gi, (lo, hi) in enumerate([(0, half), (half, spec.n_seqs)]):
        w = spec.windows[gi]
        groups.append(dict(window=w, q=inp["q"][cu[lo]:cu[hi]],
                           cu=torch.tensor([c - cu[lo] for c in cu[lo:hi + 1]], dtype=torch.int32,
                                           device=dev),
                           lens=kv.seq_lens[lo:hi].contiguous(), bt=kv.block_table[lo:hi].contiguous(),
                           rel=inp["rel"][cu[lo]:cu[hi]], out=torch.empty_like(inp["q"][cu[lo]:cu[hi]]),
                           maxq=max(q_lens[lo:hi])))
        flops += 4 * spec.Hq * spec.D * sum(sum(min(i + 1, w) if w else i + 1 for i in range(L))
                                            for L in q_lens[lo:hi])

    def step():
        for g in groups:
            fk.attn_fp8_varlen_prefill_per_token(cache, g["q"], g["cu"], g["lens"], g["bt"],
                                                 g["maxq"], 1.0, ks, vs, rel_bias=g["rel"],
                                                 window=g["window"], out=g["out"])
    ms = time_steps(step, steps, warmup, world)
    fp8_peak = 2.0 * peaks()["bf16_tflops"]
    return {"workload": spec.name + "_per_token_scales", "ms_per_step": ms,
            "tflops": flops / ms / 1e9,
            "roofline": {"bound": "tensor", "achieved": flops / ms / 1e9, "peak": fp8_peak,
                         "unit": "TFLOP/s", "frac": flops / ms / 1e9 / fp8_peak}}


def bench_chunked_prefill(fk, dev, steps, warmup, world, cpu_budget=0.0):
    """One 4,096-query chunk attending over 65,536 keys (a cached prefix)."""
    spec = workloads.PREFILL_CHUNK_64K
    inp = workloads.make_prefill(spec, device=dev, seed=0)
    kv = inp["kv"]
    cache = fk.KVCache.empty(kv.num_blocks, kv.block_size, spec.Hkv, spec.D, device=dev)
    fk.kv_store_e4m3(cache, kv.k, kv.v, kv.slot_mapping, 1.0, 1.0)
    out = torch.empty_like(inp["q"])
    maxq = max(inp["q_lens"])
    pairs = sum(sum(kl - ql + i + 1 for i in range(ql))
                for ql, kl in zip(inp["q_lens"], inp["k_lens"]))
    flops = 4 * spec.Hq * spec.D * pairs

    def step():
        fk.attn_fp8_varlen_prefill(cache, inp["q"], inp["cu_seqlens_q"], kv.seq_lens,
                                   kv.block_table, maxq, 1.0, 1.0, 1.0, rel_bias=inp["rel"],
                                   window=0, out=out)
    ms = time_steps(step, steps, warmup, world)
    fp8_peak = 2.0 * peaks()["bf16_tflops"]
    res = {"workload": spec.name, "ms_per_step": ms, "tflops": flops / ms / 1e9,
           "roofline": {"bound": "tensor", "achieved": flops / ms / 1e9, "peak": fp8_peak,
                        "unit": "TFLOP/s", "frac": flops / ms / 1e9 / fp8_peak}}
    if cpu_budget > 0:
        res["cpu_baseline"] = oracle_prefill_baseline(spec, inp, [(0, 0)], cpu_budget)
    return res


def bench_store_and_bands(fk, dev, steps, warmup, world, cpu_budget=0.0):
    """Quant-on-store of the whole 64-sequence pool (~1.05-1.1M tokens) and the band
    counters over its V, each against the measured HBM bandwidth."""
    spec = workloads.DECODE_32K
    inp = workloads.make_decode(spec, device=dev, seed=0)
    kv = inp["kv"]
    cache = fk.KVCache.empty(kv.num_blocks, kv.block_size, spec.Hkv, spec.D, device=dev)
    elems = kv.k.shape[0] * spec.Hkv * spec.D
    counts = torch.zeros(fk.BAND_COUNTS_BYTES, dtype=torch.uint8, device=dev)
    hbm = peaks()["hbm_gbs"]
    res = []
    for name, fn, nbytes in (
            ("kv_store_e4m3 of the 64-sequence pool (K and V)",
             lambda: fk.kv_store_e4m3(cache, kv.k, kv.v, kv.slot_mapping, 1.0, 3.0),
             elems * 2 * (2 + 1)),
            ("kv_band_counts over the pool's V at scale 3",
             lambda: fk.kv_band_counts(kv.v, 3.0, counts=counts), elems * 2)):
        ms = time_steps(fn, steps, warmup, world)
        gbs = nbytes / ms / 1e6
        res.append({"workload": name, "ms_per_step": ms, "gbs": gbs,
                    "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                                 "frac": gbs / hbm}})
    if cpu_budget > 0:
        res[0]["cpu_baseline"], res[1]["cpu_baseline"] = oracle_store_band_baselines(
            kv, spec, cpu_budget)
    return res


def oracle_store_band_baselines(kv, spec, budget_s):
    """The oracle's store (quantize and scatter, K and V) and band counters
    (over V at scale 3) on the pool's first tokens, in chunks of 4,096 tokens
    until about budget_s of CPU time each; GB/s over the same algorithmic
    bytes as the GPU lines (3 bytes per stored element, 2 per counted one)."""
    import oracle
    bits = workloads.bf16_bits
    cores = oracle.num_threads()
    row = spec.Hkv * spec.D
    ck = np.zeros((kv.num_blocks, spec.Hkv, kv.block_size, spec.D), dtype=np.uint8)
    cv = np.zeros_like(ck)
    out = []
    for what in ("store", "bands"):
        t_total, tokens, c0 = 0.0, 0, 0
        while t_total < budget_s and c0 < kv.k.shape[0]:
            c1 = min(c0 + 4096, kv.k.shape[0])
            vb = bits(kv.v[c0:c1])
            if what == "store":
                kb = bits(kv.k[c0:c1])
                sm = kv.slot_mapping[c0:c1].cpu().numpy()
                t0 = time.perf_counter()
                oracle.kv_store(ck, cv, kb, vb, sm, 1.0, 3.0, kv.block_size)
            else:
                t0 = time.perf_counter()
                oracle.band_counts(vb, 3.0)
            t_total += time.perf_counter() - t0
            tokens += c1 - c0
            c0 = c1
        nbytes = tokens * row * (2 * 3 if what == "store" else 2)
        out.append(cpu_line(nbytes / t_total / 1e9, "GB/s", 1,
                            "the pool's first %d tokens (%s), %.1f s of CPU time, one thread" %
                            (tokens, "K and V" if what == "store" else "V", t_total)))
    return out


def bench_decode_per_token(fk, dev, steps, warmup, world, cpu_budget=0.0):
    """The 64-sequence decode over a cache with per-token scales (written by
    kv_store_e4m3_per_token): KV bytes plus 4 bytes of K and V scale per key
    and KV head."""
    spec = workloads.DECODE_32K
    inp = workloads.make_decode(spec, device=dev, seed=0)
    kv = inp["kv"]
    cache = fk.KVCache.empty(kv.num_blocks, kv.block_size, spec.Hkv, spec.D, device=dev)
    ks = torch.empty((kv.num_blocks, spec.Hkv, kv.block_size), dtype=torch.float32, device=dev)
    vs = torch.empty_like(ks)
    fk.kv_store_e4m3_per_token(cache, kv.k, kv.v, kv.slot_mapping, ks, vs)
    q, rel = inp["q"], inp["rel"]
    out = torch.empty_like(q)
    n = fk.decode_workspace_size(q.shape[0], spec.Hq, spec.Hkv, spec.D, kv.max_blocks,
                                 kv.block_size, 0, 0)
    ws = torch.empty(n, dtype=torch.uint8, device=dev)
    keys = sum(inp["lens"]) * spec.Hkv
    nbytes = keys * (2 * spec.D + 8) + 2 * q.numel() * 2 + rel.numel() * 2

    def step():
        fk.paged_attn_fp8_decode_per_token(cache, q, kv.block_table, kv.seq_lens, 1.0, ks, vs,
                                           rel_bias=rel, out=out, workspace=ws)
    ms = time_steps(step, steps, warmup, world)
    gbs = nbytes / ms / 1e6
    hbm = peaks()["hbm_gbs"]
    res = {"workload": spec.name + "_per_token_scales", "ms_per_step": ms, "gbs": gbs,
           "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                        "frac": gbs / hbm}}
    if cpu_budget > 0:
        res["cpu_baseline"] = oracle_per_token_baseline(spec, inp, cpu_budget)
    return res


def oracle_per_token_baseline(spec, inp, budget_s):
    """The oracle's per-token store and attention (or_quantize_per_token,
    or_attend_row_pt) on whole sequences, one KV head at a time with its
    query heads, until about budget_s of CPU time; GB/s over the sample's KV
    and scale bytes."""
    import oracle
    bits = workloads.bf16_bits
    kv = inp["kv"]
    D, G = spec.D, spec.Hq // spec.Hkv
    starts = kv.tok_start.cpu().tolist()
    t_total, nbytes, units = 0.0, 0, 0
    for b, L in enumerate(inp["lens"]):
        for kvh in range(spec.Hkv):
            kb = bits(kv.k[starts[b]:starts[b] + L, kvh])
            vb = bits(kv.v[starts[b]:starts[b] + L, kvh])
            qb = [bits(inp["q"][b, kvh * G + g]) for g in range(G)]
            rb = [bits(inp["rel"][b, kvh * G + g]) for g in range(G)]
            t0 = time.perf_counter()
            k8, sk = oracle.quantize_per_token(kb, D)
            v8, sv = oracle.quantize_per_token(vb, D)
            for g in range(G):
                oracle.attend_row_pt(oracle.quantize(qb[g], 1.0), k8, v8, sk, sv, L - 1,
                                     1 / math.sqrt(D), 1.0, bias=rb[g])
            t_total += time.perf_counter() - t0
            nbytes += L * (2 * D + 8)
            units += 1
            if t_total >= budget_s:
                return cpu_line(nbytes / t_total / 1e9, "GB/s", 1,
                                "%d (sequence, KV head) pairs with their %d query heads, %.1f s of"
                                " CPU time, one thread" % (units, G, t_total))
    return cpu_line(nbytes / t_total / 1e9, "GB/s", 1, "%d (sequence, KV head) pairs, %.1f s" %
                    (units, t_total))


def bench_decode_extra(fk, spec, dev, steps, warmup, world, calibrate=False,
                       scales=(1.0, 1.0, 1.0), label=None, cpu_budget=0.0, cpu_max_keys=None):
    run = DecodeRun(fk, spec, dev, calibrate=calibrate, scales=scales)
    ms = time_steps(run.step, steps, warmup, world)
    dms = time_steps(run.decode, steps, warmup, world)
    bms = time_steps(run.bound.run, steps, warmup, world)
    hbm = peaks()["hbm_gbs"]
    dgbs = run.decode_bytes / dms / 1e6
    bgbs = run.decode_bytes / bms / 1e6
    res = {"workload": label or spec.name, "ms_per_step": ms, "gbs": run.step_bytes / ms / 1e6,
           "decode_ms": dms, "decode_gbs": dgbs, "decode_bound_ms": bms, "decode_bound_gbs": bgbs,
           "scales": list(run.scales), "window": spec.window,
           "roofline": {"bound": "hbm", "achieved": bgbs, "peak": hbm, "unit": "GB/s",
                        "frac": bgbs / hbm, "frac_of_nominal_8tbs": bgbs / 8000.0,
                        "kernel": "paged_attn_fp8_decode through DecodeStep.run (decode + split "
                                  "merge; the one-shot call's figure is decode_gbs)"}}
    if cpu_budget > 0:
        res["cpu_baseline"] = oracle_decode_baseline(spec, run.inp, run.scales, cpu_budget,
                                                     cpu_max_keys)
    del run
    torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extra", action="store_true", help="skip the secondary workloads")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--settle-s", type=float, default=0.6,
                    help="seconds of untimed steps before the timed ones, for the clock samples")
    ap.add_argument("--profile-decode", type=int, default=0, metavar="B",
                    help="profiling case: only the decode call of the 32K workload cut to B "
                         "sequences (still larger than L2), no JSON contract line")
    ap.add_argument("--profile-prefill", type=int, default=0, metavar="GROUP",
                    help="profiling case: only the prefill call of group GROUP-1 (1 = the "
                         "causal sequences, 2 = the 512-window ones) of the prefill chunk")
    ap.add_argument("--only-extra", default="",
                    help="run only the named secondary workload (per_token_decode, "
                         "per_token_prefill, window_decode) and print its JSON")
    ap.add_argument("--profile-store", action="store_true",
                    help="profiling case: only the quant-on-store of the 64-sequence pool and the "
                         "band counters over its V, no JSON contract line")
    args = ap.parse_args()
    rank, world = dist_setup(args.gpus)
    if args.only_extra:
        import dataclasses
        import fp8_e4m3_kv_gb300 as fk
        dev = torch.device("cuda", torch.cuda.current_device())
        spec = workloads.DECODE_32K
        fn = {"per_token_decode": lambda: bench_decode_per_token(fk, dev, args.steps, args.warmup,
                                                                 world),
              "per_token_prefill": lambda: bench_prefill_per_token(fk, dev, args.steps,
                                                                   args.warmup, world),
              "window_decode": lambda: bench_decode_extra(
                  fk, dataclasses.replace(spec, window=512), dev, args.steps, args.warmup, world,
                  label=spec.name + "_window512")}[args.only_extra]
        print(json.dumps(fn()))
        return
    if args.profile_store:
        import fp8_e4m3_kv_gb300 as fk
        dev = torch.device("cuda", torch.cuda.current_device())
        print(json.dumps(bench_store_and_bands(fk, dev, args.steps, args.warmup, world)))
        return
    if args.profile_prefill:
        import fp8_e4m3_kv_gb300 as fk
        dev = torch.device("cuda", torch.cuda.current_device())
        res = bench_prefill(fk, dev, args.steps, args.warmup, world,
                            only_group=args.profile_prefill - 1)
        print(json.dumps(res))
        return
    if args.profile_decode:
        import dataclasses
        import fp8_e4m3_kv_gb300 as fk
        spec = dataclasses.replace(workloads.DECODE_32K, B=args.profile_decode)
        run = DecodeRun(fk, spec, torch.device("cuda", torch.cuda.current_device()))
        ms = time_steps(run.decode, args.steps, args.warmup, world)
        print(json.dumps({"profile_case": spec.name, "seqs": spec.B, "decode_ms": ms,
                          "decode_bytes": run.decode_bytes,
                          "decode_gbs": run.decode_bytes / ms / 1e6}))
        return
    spec = workloads.DECODE_32K
    cfg = {"workload": spec.name, "seqs": spec.B, "q_heads": spec.Hq, "kv_heads": spec.Hkv,
           "head_dim": spec.D, "block_size": spec.block_size,
           "context": "U[%d,%d]" % (spec.ctx_lo, spec.ctx_hi), "rel_extent": spec.rel_extent,
           "l2": "inputs larger than L2 (~1.1 GB of fp8 KV read per step)",
           "parallelism": "replicas" if world > 1 else "single"}

    if args.impl == "reference":
        if rank != 0:
            return
        # a 4-sequence draw of the same workload recipe (the oracle cannot
        # hold the whole 64-sequence pool in a few minutes of CPU time)
        inp = workloads.make_decode(spec, device="cpu", seed=0, B=4)
        per_step, step_ms = [], []
        desc = None
        for _ in range(max(1, args.steps)):
            gbs, seqs, t, cores = oracle_decode_sample(spec, inp, (1.0, 1.0, 1.0),
                                                       budget_s=max(2.0, 60.0 / max(1, args.steps)))
            per_step.append(gbs)
            step_ms.append(t * 1e3)
            desc = "%d whole sequences (all 32 q heads) of the workload per step, %.1f s" % (seqs, t)
        v = statistics.median(per_step)
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": statistics.median(step_ms), "higher_is_better": True,
                "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": cfg,
                "cpu_baseline": {"value": v, "unit": "GB/s", "cores": cores, "kind": "oracle",
                                 "sample": desc},
                "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import fp8_e4m3_kv_gb300 as fk
    dev = torch.device("cuda", torch.cuda.current_device())
    pk = peaks()
    run = DecodeRun(fk, spec, dev)
    # warm-up + timed region, clocks sampled during it; the untimed load
    # before the timed steps lets the sampler see the clocks under this load
    # even when K steps last only milliseconds
    with ClockSampler(dev.index) as clk:
        load_until = time.time() + args.settle_s
        while time.time() < load_until:
            for _ in range(50):
                run.step()
            torch.cuda.synchronize()
        ms = time_steps(run.step, args.steps, args.warmup, world)
        # the dominant kernel's call, timed alone on its stream
        dms = time_steps(run.decode, args.steps, args.warmup, world)
        # the same step as separate calls, for comparison
        sep_ms = time_steps(run.step_separate, args.steps, args.warmup, world)
    clocks = clk.summary()
    value = run.step_bytes * world / ms / 1e6          # GB/s over all ranks
    achieved = run.decode_bytes / dms / 1e6
    e2e, h2d, d2h = e2e_decode(run, max(3, args.steps // 2), args.warmup, world)
    e2e_ms = e2e["graph"]
    line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
            "data": "synthetic", "config": cfg,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"],
                         "unit": "GB/s", "frac": achieved / pk["hbm_gbs"],
                         "frac_of_nominal_8tbs": achieved / 8000.0,
                         "traffic": decode_traffic_bytes(),
                         "kernel": "paged_attn_fp8_decode (decode + split merge)",
                         "peak_source": pk["source"]},
            "e2e": {"value": run.step_bytes * world / e2e_ms / 1e6, "unit": "GB/s",
                    "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h,
                    "launch": "DecodeStep.cuda_graph: one graph replay per step (copy in, "
                              "store + decode, read back), then a host sync",
                    "eager": {"value": run.step_bytes * world / e2e["eager"] / 1e6,
                              "ms_per_step": e2e["eager"],
                              "launch": "the copy, DecodeStep.run and the read back issued "
                                        "one by one"}},
            "gpu_launches": run.launches_per_step * args.steps,
            "separate_calls": {"ms_per_step": sep_ms, "value": run.step_bytes * world / sep_ms / 1e6,
                               "launches_per_step": 4},
            "clocks": clocks}
    scales = run.scales
    inp_cpu = None
    if rank == 0 and not args.no_cpu:
        inp_cpu = run.inp
    del run
    torch.cuda.empty_cache()
    if not args.no_extra:
        import dataclasses
        extra = []
        cb = 5.0 if (rank == 0 and not args.no_cpu) else 0.0   # CPU seconds per extra
        for fn in (lambda: bench_prefill(fk, dev, args.steps, args.warmup, world, cpu_budget=cb),
                   lambda: bench_chunked_prefill(fk, dev, max(3, args.steps // 4), args.warmup,
                                                 world, cpu_budget=cb),
                   lambda: bench_prefill_per_token(fk, dev, args.steps, args.warmup, world),
                   lambda: bench_store_and_bands(fk, dev, args.steps, args.warmup, world,
                                                 cpu_budget=cb),
                   lambda: bench_decode_per_token(fk, dev, args.steps, args.warmup, world,
                                                  cpu_budget=cb),
                   lambda: bench_decode_extra(fk, dataclasses.replace(spec, window=512), dev,
                                              args.steps, args.warmup, world,
                                              label=spec.name + "_window512", cpu_budget=cb),
                   lambda: bench_decode_extra(fk, spec, dev, args.steps, args.warmup, world,
                                              scales=(1.0, 1.0, 3.0),
                                              label=spec.name + "_vscale3", cpu_budget=cb),
                   lambda: bench_decode_extra(fk, workloads.DECODE_128K_CAL, dev, args.steps,
                                              args.warmup, world, calibrate=True, cpu_budget=cb,
                                              cpu_max_keys=8192),
                   lambda: bench_decode_extra(fk, workloads.DECODE_1M, dev, args.steps,
                                              args.warmup, world, cpu_budget=cb,
                                              cpu_max_keys=65536)):
            try:
                r = fn()
                extra.extend(r if isinstance(r, list) else [r])
            except Exception as e:  # noqa: BLE001
                extra.append({"error": repr(e)[:300]})
            torch.cuda.empty_cache()
        line["extra"] = extra
    if rank == 0 and inp_cpu is not None:
        gbs, seqs, t, cores = oracle_decode_sample(spec, inp_cpu, scales, budget_s=15.0)
        line["cpu_baseline"] = {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle",
                                "sample": "%d whole sequences (all 32 q heads, float64) of the "
                                          "workload, %.1f s of CPU time" % (seqs, t)}
    if rank == 0:
        print(json.dumps(line))


if __name__ == "__main__":
    main()
