#!/usr/bin/env python3
"""Throughput of the DSA sparse-attention hot path on GB300.

A step is one pass of the path over one batch of synthetic input:
  decode workloads : index score -> top-K -> sparse attention (decode)
  prefill workload : index score -> top-K -> sparse attention (prefill)
The default workload is "dec-batch" (32 sequences, L ~ U[8192, 32768], latent
64x576 KV, FP8 indexer, top-K 2048); its metric is decode queries/s.  The
prefill workload (16384 tokens, same shapes) is measured in the same run and
reported under "prefill" (tokens/s) unless --secondary is empty.

Timing: W untimed warm-up steps; the step (and each of its three stages) is
then captured once into a CUDA graph; K timed replays follow.  Before each
timed replay L2 is flushed outside the timed region: a 512 MiB buffer is
written, then a 256 MiB buffer is read, so that the dirty lines the write
leaves in L2 are written back before the step starts instead of during its
first kernel (the step starts from a cold and clean L2); each replay is bracketed by CUDA events on the stream the kernels run
on, with a barrier and a synchronize on both sides of the timed loop; the
reported time is the max over ranks.  Per-stage times come from the stage
graphs, each replayed on its own right after the flush.  With N GPUs (torchrun) every rank runs its own batch
(weak scaling, no data-path collective).

--impl reference times the CPU oracle (test infrastructure, one thread) on a
bounded sample of the same workload.
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
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FLUSH_BYTES = 512 << 20       # written (more than the 129 MB of L2)
FLUSH_READ_BYTES = 256 << 20  # then read, which writes the dirty lines back
L2_NOTE = "flushed: 512 MiB written, then 256 MiB read, before every timed step (cold, clean L2)"


class L2Flush:
    """Evicts L2 between timed steps: a write of a buffer larger than L2, then a
    read of another one, so that no dirty line of the write is left for the
    timed kernels to write back."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.r = torch.ones(FLUSH_READ_BYTES // 4, dtype=torch.float32, device=dev)
        self.acc = torch.zeros((), dtype=torch.float32, device=dev)

    def __call__(self, v=1.0):
        import torch
        self.w.fill_(float(v))
        torch.sum(self.r, dim=0, out=self.acc)


# ------------------------------------------------------------------ helpers --
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


class ClockSampler:
    """SM clock and clock-event reasons of one GPU, sampled while the timed
    region runs.  Reads NVML directly (read-only queries, as fast as the host
    thread can poll, so even a region of a few milliseconds gets samples);
    falls back to `nvidia-smi -lms 100` when NVML cannot be loaded."""

    # nvmlClocksEventReason* bits
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, cuda_index: int):
        self.cuda_index = cuda_index
        self.samples = []          # (sm_mhz, reasons bitmask)
        self.max_mhz = None
        self.proc = None
        self.lines = []
        self.nvml = None
        self.handle = None
        self._stop = threading.Event()
        self.t = None
        try:
            import ctypes
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            rc = 1
            bus = self._pci_bus_id()
            if bus:
                rc = nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h))
            if rc != 0:
                rc = nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(cuda_index), ctypes.byref(h))
            if rc != 0:
                return
            self.reason_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:   # NVML_CLOCK_SM
                self.max_mhz = float(mx.value)
            self.nvml, self.handle, self.ct = nv, h, ctypes
        except (OSError, AttributeError):
            self.nvml = None

    def _pci_bus_id(self):
        try:
            import torch
            p = torch.cuda.get_device_properties(self.cuda_index)
            return "%08X:%02X:%02X.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
        except Exception:
            return None

    def _poll(self):
        ct, nv, h = self.ct, self.nvml, self.handle
        mhz, rs = ct.c_uint(), ct.c_ulonglong()
        while not self._stop.is_set():
            if nv.nvmlDeviceGetClockInfo(h, 1, ct.byref(mhz)) == 0 and \
                    self.reason_fn(h, ct.byref(rs)) == 0:
                self.samples.append((float(mhz.value), int(rs.value)))
            time.sleep(0.0002)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def start(self):
        if self.nvml is not None:
            self.t = threading.Thread(target=self._poll, daemon=True)
            self.t.start()
            t0 = time.perf_counter()
            while not self.samples and time.perf_counter() - t0 < 1.0:
                time.sleep(0.0005)
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.cuda_index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.nvml is not None:
            self._stop.set()
            self.t.join(timeout=2)
            if not self.samples:
                return None
            reasons = sorted({nm for _, r in self.samples for b, nm in self.REASONS.items() if r & b})
            return {"sm_mhz": statistics.median(m for m, _ in self.samples),
                    "sm_max_mhz": self.max_mhz, "reasons": reasons,
                    "samples": len(self.samples), "source": "nvml"}
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "source": "nvidia-smi"}


def kernel_source_sha(names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "sparse_attention_score_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_key, src_files):
    """Per-launch DRAM bytes of a kernel from a committed ncu summary, or None if
    the kernel source changed since the counters were taken."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel_key)
    if not e or e.get("source_sha") != kernel_source_sha(src_files):
        return None
    return e.get("traffic_bytes_per_launch")


# ---------------------------------------------------------------- workloads --
PREFILL_TOKENS = None  # --prefill-tokens: a shorter prompt (profiling captures)


def workload_case(name, rank):
    import workloads as W
    # weak scaling: every rank draws its own batch
    seeds = {"dec-tiny": 0, "dec-batch": 1, "prefill": 2, "long-dec": 3, "million": 4}
    kw = {}
    if name == "prefill" and PREFILL_TOKENS:
        kw["T"] = PREFILL_TOKENS
    return W.config(name, seed=seeds[name] + 1000 * rank, **kw)


def algorithmic(case):
    """Algorithmic bytes / flops of one step (indexer keys + gathered KV rows for
    decode; tensor flops for prefill)."""
    elt_i = 1 if case.idx_dtype == "fp8" else 2
    sel = np.minimum(case.n_elig.astype(np.int64), case.K)
    kv_row = case.Dkv * 2 if case.latent else (case.Dqk + case.Dv) * 2
    idx_bytes = int(case.n_elig.astype(np.int64).sum()) * case.D_i * elt_i
    if case.kind == "decode":
        idx_bytes = int(case.seq_lens.astype(np.int64).sum()) * case.D_i * elt_i
    gather_bytes = int(sel.sum()) * kv_row
    idx_flops = 2.0 * float(case.n_elig.astype(np.int64).sum()) * case.H_i * case.D_i
    attn_flops = 2.0 * float(sel.sum()) * case.Hq * (case.Dqk + case.Dv)
    return dict(index_bytes=idx_bytes, gather_bytes=gather_bytes, index_flops=idx_flops,
                attn_flops=attn_flops)


# ------------------------------------------------------------- multi-rank --
def max_over_ranks(value, world, device):
    """The slowest rank's value (weak scaling: every rank times its own batch,
    the job takes as long as the slowest); a barrier follows, so no rank
    leaves before all have reported."""
    if world <= 1:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    torch.distributed.barrier()
    return float(t.item())


# ----------------------------------------------------------------- GPU arm --
def run_gpu(name, steps, warmup, rank, world, local_rank, do_e2e=True):
    import torch

    import sparse_attention_score_gb300 as dsa
    from workloads import device as wdev

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    case = workload_case(name, rank)
    d = wdev.upload(case, dev)
    layout = wdev.layout_of(case, d)
    kind = case.kind
    pipe = dsa.Pipeline(layout, kind=kind, Nq=case.Nq, Hq=case.Hq, Dqk=case.Dqk, Dv=case.Dv,
                        H_i=case.H_i, D_i=case.D_i, K=case.K, device=dev)
    qp = None if kind == "decode" else d.q_pos
    stream = torch.cuda.current_stream(dev)
    flush = L2Flush(dev)

    def stage_index():
        if kind == "decode":
            dsa.index_score(layout, d.q_idx, d.w, d.kidx_pool, pipe.scores, pipe.ws_index)
        else:
            dsa.index_score_prefill(layout, 0, d.q_idx, d.w, d.kidx_pool, pipe.scores,
                                    pipe.ws_index, q_pos=qp)

    def stage_topk():
        dsa.topk(pipe.scores, d.n_elig, case.K, pipe.idx, pipe.ws_topk)

    def stage_attn():
        if kind == "decode":
            dsa.sparse_attn_decode(layout, d.q, d.k_pool, d.v_pool, pipe.idx, case.sm_scale,
                                   pipe.out, pipe.lse, pipe.ws_attn)
        else:
            dsa.sparse_attn_prefill(layout, d.q, d.k_pool, d.v_pool, pipe.idx, case.sm_scale,
                                    pipe.out, pipe.lse, pipe.ws_attn, q_seq=d.q_seq,
                                    q_pos=d.q_pos)

    def step():
        stage_index()
        stage_topk()
        stage_attn()

    for _ in range(warmup):
        flush(1.0)
        step()
    torch.cuda.synchronize()
    # The step (and each stage) is captured once into a CUDA graph and
    # replayed: the timed region holds device work only, no host launch cost.
    graphs = {}
    launches_per = {}
    for name_, fn in (("step", step), ("index_score", stage_index), ("topk", stage_topk),
                      ("sparse_attn", stage_attn)):
        g_ = torch.cuda.CUDAGraph()
        n0 = dsa.launch_count()
        with torch.cuda.graph(g_):
            fn()
        launches_per[name_] = dsa.launch_count() - n0
        graphs[name_] = g_
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()

    sampler = ClockSampler(local_rank)
    sampler.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for i in range(steps):
        flush(float(i))
        ev[i][0].record(stream)
        graphs["step"].replay()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    step_ms = np.array([a_.elapsed_time(b_) for a_, b_ in ev])
    total_ms = float(step_ms.sum())
    launches = launches_per["step"] * steps
    # per-stage device time: each stage graph replayed on its own, right after
    # the L2 flush kernel (which keeps the GPU busy while the host submits the
    # replay, so no host gap lands between the events)
    stage = np.zeros((steps, 3))
    for k, name_ in enumerate(("index_score", "topk", "sparse_attn")):
        sev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for i in range(steps):
            flush(float(i))
            sev[i][0].record(stream)
            graphs[name_].replay()
            sev[i][1].record(stream)
        torch.cuda.synchronize()
        stage[:, k] = [a_.elapsed_time(b_) for a_, b_ in sev]
    status = pipe.status()
    cache_write = measure_cache_write(dsa, case, d, layout, dev, flush, steps)
    step_calls = bounded = None
    if kind == "prefill":
        step_calls = measure_prefill_steps(dsa, case, d, layout, dev, flush, steps)
    else:
        bounded = measure_bounded_index(dsa, case, d, layout, dev, flush, steps, pipe.idx.clone())

    e2e = None
    if do_e2e:
        e2e = run_e2e(case, d, pipe, steps, dev, flush)

    total_ms = max_over_ranks(total_ms, world, dev)
    return dict(case=case, total_ms=total_ms, stage_ms=stage.mean(axis=0).tolist(),
                launches=int(launches), launches_per=launches_per, clocks=clocks, status=status,
                e2e=e2e, graph=graphs["step"], cache_write=cache_write, step_calls=step_calls,
                bounded_index=bounded)


def measure_cache_write(dsa, case, d, layout, dev, flush, steps):
    """The cache write that feeds the step, timed on its own: decode appends
    each sequence's newest row, prefill stores the whole prompt.  The rows
    written are the rows already cached there (read back through the block
    table), so the cache the step reads is unchanged.  Algorithmic bytes: each
    K/V row and indexer-key row read once and written once."""
    import torch
    if case.kind == "decode":
        seq = torch.arange(case.B, dtype=torch.int32, device=dev)
        pos = (d.seq_lens - 1).to(torch.int32)
    else:
        seq = torch.zeros(case.Nq, dtype=torch.int32, device=dev)
        pos = d.q_pos.clone()
    pl, sl = pos.long(), seq.long()
    phys = d.block_table.long()[sl, pl // case.bs] * case.bs + pl % case.bs
    kv_rows = d.k_pool.view(-1, d.k_pool.shape[-1])[phys].contiguous()
    ki_rows = d.kidx_pool.view(-1, d.kidx_pool.shape[-1])[phys].contiguous()
    ws = dsa.workspace(dsa.cache_write_workspace_size(), device=dev)
    stream = torch.cuda.current_stream(dev)

    def call():
        dsa.cache_write(layout, seq, pos, ws, kv_new=kv_rows, kv_pool=d.k_pool, kidx_new=ki_rows,
                        kidx_pool=d.kidx_pool)

    for _ in range(3):
        call()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for i in range(steps):
        flush(float(i))
        ev[i][0].record(stream)
        call()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    us = float(np.mean([a_.elapsed_time(b_) for a_, b_ in ev])) * 1e3
    n = int(seq.shape[0])
    row_bytes = kv_rows.shape[1] * kv_rows.element_size() + ki_rows.shape[1] * ki_rows.element_size()
    nbytes = 2 * n * row_bytes
    return {"rows": n, "bytes_per_row": int(row_bytes), "us": round(us, 2),
            "achieved_gbs": round(nbytes / (us * 1e-6) / 1e9, 1),
            "status": dsa.get_status(ws)}


def measure_bounded_index(dsa, case, d, layout, dev, flush, steps, ref_idx):
    """The decode indexer with block-level bounds (dsa_index_score_bounded): the
    bound pool built once for every cached page (timed), then the bounded
    scoring timed like a stage, the tiles it left out, and whether dsa_topk over
    its row selects what the step selected."""
    import torch
    kb = torch.zeros((case.num_blocks, 2, case.D_i), dtype=d.kidx_pool.dtype, device=dev)
    wsb = dsa.workspace(dsa.index_bounds_update_workspace_size(), device=dev)
    stream = torch.cuda.current_stream(dev)
    dsa.index_bounds_update(layout, d.kidx_pool, kb, wsb)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    flush(0.5)
    e0.record(stream)
    dsa.index_bounds_update(layout, d.kidx_pool, kb, wsb)
    e1.record(stream)
    torch.cuda.synchronize()
    build_us = e0.elapsed_time(e1) * 1e3
    ld = (int(case.seq_lens.max()) + 3) // 4 * 4
    scores = torch.empty((case.B, ld), dtype=torch.float32, device=dev)
    ws = dsa.workspace(dsa.index_score_bounded_workspace_size(case.B, case.H_i, case.D_i, ld,
                                                              case.K), device=dev)

    def call():
        dsa.index_score_bounded(layout, d.q_idx, d.w, d.kidx_pool, kb, case.K, scores, ws)

    for _ in range(2):
        call()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for i in range(steps):
        flush(float(i))
        ev[i][0].record(stream)
        call()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    us = float(np.mean([a_.elapsed_time(b_) for a_, b_ in ev])) * 1e3
    skipped, total = dsa.index_bounded_stats(ws)
    idx = torch.empty((case.B, case.K), dtype=torch.int32, device=dev)
    wt = dsa.workspace(dsa.topk_workspace_size(case.B, ld, case.K), device=dev)
    dsa.topk(scores, d.n_elig, case.K, idx, wt)
    torch.cuda.synchronize()
    return {"tiles_left_out": skipped, "tiles": total, "us": round(us, 2),
            "bounds_build_us": round(build_us, 2),
            "idx_equal": bool(torch.equal(idx, ref_idx)),
            "status": dsa.get_status(ws) | dsa.get_status(wsb),
            "api": "dsa_index_score_bounded (bound pool from dsa_index_bounds_update)"}


def measure_prefill_steps(dsa, case, d, layout, dev, flush, steps):
    """The whole prefill step through one binding call, two ways: the staged
    dsa_prefill_step (the caller's [Nq][ld] score matrix between the indexer
    and top-K) and dsa_prefill_step_chunked (one chunk of scores at a time in
    an L2-sized workspace scratch).  Both include the cache write of the
    prompt's rows (the rows already cached, read back through the block
    table, so the cache is unchanged); the index sets must agree."""
    import torch
    pl = d.q_pos.long()
    phys = d.block_table.long()[0, pl // case.bs] * case.bs + pl % case.bs
    kv_rows = d.k_pool.view(-1, d.k_pool.shape[-1])[phys].contiguous()
    ki_rows = d.kidx_pool.view(-1, d.kidx_pool.shape[-1])[phys].contiguous()
    Nq, ld, K = case.Nq, int(case.n_elig.max()), case.K
    ld = (ld + 3) // 4 * 4
    scores = torch.empty((Nq, ld), dtype=torch.float32, device=dev)
    outs = {m: (torch.empty((Nq, K), dtype=torch.int32, device=dev),
                torch.empty((Nq, case.Hq, case.Dv), dtype=torch.bfloat16, device=dev),
                torch.empty((Nq, case.Hq), dtype=torch.float32, device=dev))
            for m in ("staged", "chunked")}
    ws_s = dsa.workspace(dsa.prefill_step_workspace_size(Nq, case.H_i, case.D_i, ld, case.Hq,
                                                         case.Dqk, case.Dv, K), device=dev)
    ws_c = dsa.workspace(dsa.prefill_step_chunked_workspace_size(
        Nq, case.H_i, case.D_i, ld, case.Hq, case.Dqk, case.Dv, K, 0), device=dev)
    common = (layout, 0, d.q_pos, d.n_elig, kv_rows, d.k_pool, ki_rows, d.kidx_pool, d.q_idx,
              d.w, d.q, K, case.sm_scale)

    def staged():
        i, o, l_ = outs["staged"]
        dsa.prefill_step(*common, scores, i, o, l_, ws_s)

    def chunked():
        i, o, l_ = outs["chunked"]
        dsa.prefill_step_chunked(*common, ld, i, o, l_, ws_c)

    stream = torch.cuda.current_stream(dev)
    res = {}
    for name_, fn in (("staged", staged), ("chunked", chunked)):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        for i in range(steps):
            flush(float(i))
            ev[i][0].record(stream)
            fn()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        res[name_ + "_ms"] = round(float(np.mean([a_.elapsed_time(b_) for a_, b_ in ev])), 4)
    res["score_bytes_staged"] = int(Nq * ld * 4)
    res["workspace_bytes_chunked"] = int(ws_c.numel())
    res["idx_equal"] = bool(torch.equal(outs["staged"][0], outs["chunked"][0]))
    res["status"] = dsa.get_status(ws_s) | dsa.get_status(ws_c)
    res["api"] = "dsa_prefill_step vs dsa_prefill_step_chunked, one call each, cache write included"
    del scores
    return res


def _e2e_inputs(case, dev, extra=None):
    """The step's inputs (indexer queries, weights, block table, lengths, any
    `extra` arrays, then the attention queries) as one packed pinned host
    buffer, its device twin, views of the twin shaped as each input (the
    stages read those), and the offset where the attention queries start."""
    import torch
    parts = {
        "q_idx": (case.q_idx, torch.bfloat16 if case.idx_dtype == "bf16" else torch.uint8),
        "w": (case.w, torch.float32),
        "block_table": (case.block_table, torch.int32),
        "seq_lens": (case.seq_lens, torch.int32),
    }
    parts.update(extra or {})
    parts["q"] = (case.q, torch.bfloat16)
    offs, total = {}, 0
    for k, (arr, _) in parts.items():
        offs[k] = total
        total += (arr.nbytes + 255) // 256 * 256
    hbuf = torch.zeros(total, dtype=torch.uint8).pin_memory()
    for k, (arr, _) in parts.items():
        raw = torch.from_numpy(np.ascontiguousarray(arr).view(np.uint8).reshape(-1))
        hbuf[offs[k]:offs[k] + raw.numel()].copy_(raw)
    dbuf = torch.empty(total, dtype=torch.uint8, device=dev)
    dbuf.copy_(hbuf)
    v = {k: dbuf[offs[k]:offs[k] + arr.nbytes].view(dt).view(arr.shape)
         for k, (arr, dt) in parts.items()}
    return hbuf, dbuf, v, total, offs["q"]


def run_e2e(case, d, pipe, steps, dev, flush):
    """The step end to end through the public API with host buffers, timed
    two ways.  Every timed step holds: the H2D copy of the step's inputs from
    pinned memory (one packed buffer), the three stages, and the D2H copy of
    the attention output into pinned memory; the paged KV and indexer-key
    caches are persistent device state and stay resident.  Before each step
    L2 is flushed and the device synchronised, so host-side costs are not
    hidden behind the flush.
      calls : one H2D copy, then the three binding calls made every step
              (ctypes marshalling, operand checks and kernel launches inside
              the timed region);
      graph : the copies and the three calls captured once into a CUDA graph,
              replayed each step; in it the indexer's inputs are copied first
              and the attention queries (most of the bytes, read by the
              attention stage only) on a second stream, beside the indexer
              and the top-K, the attention waiting for them.  (Issuing that
              second stream from Python every step cost more host time than
              the overlap saved.)"""
    import torch

    import sparse_attention_score_gb300 as dsa
    hbuf, dbuf, v, total, split = _e2e_inputs(case, dev)
    layout = dsa.PagedLayout(v["block_table"], v["seq_lens"], case.bs, case.num_blocks,
                             case.max_len)
    out_host = torch.empty(pipe.out.shape, dtype=pipe.out.dtype).pin_memory()
    d2h = out_host.numel() * out_host.element_size()
    stream = torch.cuda.current_stream(dev)
    side = torch.cuda.Stream(dev)
    q_ready = torch.cuda.Event()
    ref_out = pipe.out.clone()  # the device-resident step's output on the same inputs

    def step_body(overlap):
        cur = torch.cuda.current_stream(dev)
        if overlap:
            side.wait_stream(cur)  # the side copy starts after everything queued before it
            dbuf[:split].copy_(hbuf[:split], non_blocking=True)
            with torch.cuda.stream(side):
                dbuf[split:].copy_(hbuf[split:], non_blocking=True)
                q_ready.record(side)
        else:
            dbuf.copy_(hbuf, non_blocking=True)
        if case.kind == "decode":
            dsa.index_score(layout, v["q_idx"], v["w"], d.kidx_pool, pipe.scores, pipe.ws_index)
            dsa.topk(pipe.scores, v["seq_lens"], case.K, pipe.idx, pipe.ws_topk)
            if overlap:
                cur.wait_event(q_ready)
            dsa.sparse_attn_decode(layout, v["q"], d.k_pool, d.v_pool, pipe.idx, case.sm_scale,
                                   pipe.out, pipe.lse, pipe.ws_attn)
        else:
            dsa.index_score_prefill(layout, 0, v["q_idx"], v["w"], d.kidx_pool, pipe.scores,
                                    pipe.ws_index, q_pos=d.q_pos)
            dsa.topk(pipe.scores, d.n_elig, case.K, pipe.idx, pipe.ws_topk)
            if overlap:
                cur.wait_event(q_ready)
            dsa.sparse_attn_prefill(layout, v["q"], d.k_pool, d.v_pool, pipe.idx, case.sm_scale,
                                    pipe.out, pipe.lse, pipe.ws_attn, q_seq=d.q_seq,
                                    q_pos=d.q_pos)
        out_host.copy_(pipe.out, non_blocking=True)

    step_body(False)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step_body(True)
    torch.cuda.synchronize()

    def step_calls():
        step_body(False)

    def step_graph():
        g.replay()

    units = case.Nq if case.kind == "prefill" else case.B
    res = {}
    for key, fn in (("calls", step_calls), ("graph", step_graph)):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        tot = 0.0
        for _ in range(steps):
            flush(2.0)
            torch.cuda.synchronize()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            tot += a.elapsed_time(b)
        res[key] = {"value": units * steps / (tot / 1e3), "unit": unit_of(case),
                    "h2d_bytes_per_step": int(total), "d2h_bytes_per_step": int(d2h),
                    "h2d_copies_per_step": 2 if key == "graph" else 1, "d2h_copies_per_step": 1,
                    "out_equal": bool(torch.equal(out_host, ref_out.cpu()))}
    if case.kind == "decode":
        res["step"] = run_e2e_decode_step(case, d, pipe, steps, dev, flush, units, ref_out)
    res["calls"]["api"] = ("index_score, topk, sparse_attn called through the binding every "
                           "step")
    res["graph"]["api"] = ("the same calls and the copies captured once in a CUDA graph, "
                           "replayed per step, Q copied on a second stream beside the indexer "
                           "and top-K")
    return res


def run_e2e_decode_step(case, d, pipe, steps, dev, flush, units, ref_out):
    """The decode step as the single call a decoding loop makes
    (dsa_decode_step: append each sequence's new K/V and indexer-key rows at
    its last position, then index, select and attend), end to end with host
    buffers like run_e2e's calls variant.  The rows appended are the ones
    already cached at those positions, so the cache, and so the output, stay
    those of the other variants; the step does the cache write on top of
    their work."""
    import torch

    import sparse_attention_score_gb300 as dsa
    L = case.seq_lens.astype(np.int64)
    pages = case.block_table[np.arange(case.B), (L - 1) // case.bs]
    rows = (L - 1) % case.bs
    idx_t = torch.bfloat16 if case.idx_dtype == "bf16" else torch.uint8
    extra = {"k_new": (np.ascontiguousarray(case.k_pool[pages, rows]), torch.bfloat16),
             "kidx_new": (np.ascontiguousarray(case.kidx_pool[pages, rows]), idx_t)}
    if not case.latent:
        extra["v_new"] = (np.ascontiguousarray(case.v_pool[pages, rows]), torch.bfloat16)
    hbuf, dbuf, v, total, _ = _e2e_inputs(case, dev, extra)
    layout = dsa.PagedLayout(v["block_table"], v["seq_lens"], case.bs, case.num_blocks,
                             case.max_len)
    out_host = torch.empty(pipe.out.shape, dtype=pipe.out.dtype).pin_memory()
    d2h = out_host.numel() * out_host.element_size()
    ws = dsa.workspace(dsa.decode_step_workspace_size(case.B, case.H_i, case.D_i,
                                                      pipe.scores.shape[1], case.Hq, case.Dqk,
                                                      case.Dv, case.K), device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        dbuf.copy_(hbuf, non_blocking=True)
        dsa.decode_step(layout, v["k_new"], d.k_pool, v["kidx_new"], d.kidx_pool, v["q_idx"],
                        v["w"], v["q"], case.K, case.sm_scale, pipe.scores, pipe.idx, pipe.out,
                        pipe.lse, ws, v_new=v.get("v_new"),
                        v_pool=None if case.latent else d.v_pool)
        out_host.copy_(pipe.out, non_blocking=True)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    tot = 0.0
    for _ in range(steps):
        flush(2.0)
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step()
        b.record(stream)
        b.synchronize()
        tot += a.elapsed_time(b)
    return {"value": units * steps / (tot / 1e3), "unit": unit_of(case),
            "h2d_bytes_per_step": int(total), "d2h_bytes_per_step": int(d2h),
            "h2d_copies_per_step": 1, "d2h_copies_per_step": 1,
            "out_equal": bool(torch.equal(out_host, ref_out.cpu())),
            "status": dsa.get_status(ws),
            "api": "dsa_decode_step, one call per step (cache append + index + top-K + "
                   "attention)"}


def unit_of(case):
    return "tokens/s" if case.kind == "prefill" else "queries/s"


def metric_of(case):
    return "prefill tokens/sec" if case.kind == "prefill" else "decode queries/sec"


def roofline_of(res, peaks):
    """Roofline of the dominant kernel and of the whole step."""
    case = res["case"]
    alg = algorithmic(case)
    st = res["stage_ms"]  # [index, topk, attn] ms per step (avg)
    if case.kind == "decode":
        cands = {
            "index_score": (alg["index_bytes"], st[0], ["index_score.cu", "index_tc.cu"]),
            "sparse_attn": (alg["gather_bytes"], st[2], ["attn.cu", "attn_tc.cu"]),
        }
        dom = max(cands, key=lambda k: cands[k][1])
        nbytes, ms, srcs = cands[dom]
        ach = nbytes / (ms / 1e3) / 1e9
        roof = {"bound": "hbm", "kernel": dom, "achieved": round(ach, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(ach / peaks["hbm_gbs"], 4),
                "traffic": ncu_traffic(f"{dom}:{case.name}", srcs),
                "peak_source": peaks["source"]}
        step_bytes = alg["index_bytes"] + alg["gather_bytes"]
        return roof, step_bytes
    cands = {
        "index_score": (alg["index_flops"], st[0], ["index_score.cu", "index_prefill_tc.cu"]),
        "sparse_attn": (alg["attn_flops"], st[2], ["attn.cu", "attn_tc.cu"]),
    }
    dom = max(cands, key=lambda k: cands[k][1])
    fl, ms, srcs = cands[dom]
    ach = fl / (ms / 1e3) / 1e12
    # FP8 indexer: the bf16 peak times the nominal fp8/bf16 ratio of 2
    peak = peaks["bf16_tflops"] * (2.0 if (dom == "index_score" and case.idx_dtype == "fp8") else 1.0)
    roof = {"bound": "tensor", "kernel": dom, "achieved": round(ach, 2), "peak": round(peak, 1),
            "unit": "TFLOP/s", "frac": round(ach / peak, 4),
            "traffic": ncu_traffic(f"{dom}:{case.name}", srcs), "peak_source": peaks["source"]}
    return roof, alg["index_flops"] + alg["attn_flops"]


# ---------------------------------------------------------------- CPU oracle --
def oracle_sample(case, budget_s=15.0, max_units=None):
    """Run the oracle over queries of the case until the budget is spent; returns
    (units processed, seconds)."""
    import oracle
    code = oracle.BF16 if case.idx_dtype == "bf16" else oracle.FP8_E4M3
    t0 = time.perf_counter()
    done = 0
    order = np.arange(case.Nq)
    if case.kind == "prefill":
        order = np.random.default_rng(0).permutation(case.Nq)
    for r in order:
        rr = np.array([r])
        s = oracle.index_score(case.block_table, case.seq_lens, case.bs, case.num_blocks,
                               case.q_seq[rr], case.q_pos[rr], case.q_idx[rr], case.w[rr],
                               case.kidx_pool, code, int(case.n_elig[r]))
        idx = oracle.topk(s, case.n_elig[rr], case.K)
        oracle.sparse_attn(case.block_table, case.seq_lens, case.bs, case.num_blocks,
                           case.q_seq[rr], case.q[rr], case.k_pool, case.v_pool, idx,
                           case.sm_scale, Dv=case.Dv)
        done += 1
        if time.perf_counter() - t0 > budget_s or (max_units and done >= max_units):
            break
    return done, time.perf_counter() - t0


def host_cpu():
    """The host the oracle runs on: logical CPUs and the CPU model (lscpu's
    'Model name', else /proc/cpuinfo, else the platform string)."""
    import platform
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().startswith("Model name:"):
                model = ln.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not model and os.path.exists("/proc/cpuinfo"):
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith("model name"):
                    model = ln.split(":", 1)[1].strip()
                    break
    return {"nproc": os.cpu_count(), "cpu_model": model or platform.processor() or
            platform.machine()}


def cpu_baseline(case, budget_s):
    n, t = oracle_sample(case, budget_s)
    return {"value": n / t, "unit": unit_of(case), "cores": 1, "kind": "oracle",
            "sample": f"{n} of {case.Nq} queries of {case.name} (all three stages, fp64 C oracle, "
                      f"{t:.1f} s)", "host": host_cpu()}


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    case = workload_case(args.workload, 0)
    per_step_budget = max(1.0, args.ref_step_seconds)
    for _ in range(args.warmup):
        oracle_sample(case, per_step_budget, max_units=1)
    units, secs = 0, 0.0
    for _ in range(args.steps):
        n, t = oracle_sample(case, per_step_budget)
        units += n
        secs += t
    val = units / secs
    line = {
        "impl": "reference", "metric": metric_of(case), "value": val, "unit": unit_of(case),
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(case, world),
        "cpu_baseline": {"value": val, "unit": unit_of(case), "cores": 1, "kind": "oracle",
                         "sample": f"{units} queries of {case.name} over {args.steps} steps "
                                   f"({units / args.steps:.0f} per step)", "host": host_cpu()},
        "e2e": {"value": val, "unit": unit_of(case), "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------- main --
def config_of(case, world):
    c = {"workload": case.name, "batch": case.B, "queries": case.Nq,
         "seq_lens": ("U[8192,32768]" if case.name == "dec-batch" else
                      sorted(set(int(x) for x in case.seq_lens))[:8]),
         "heads": case.Hq, "dqk": case.Dqk, "dv": case.Dv, "latent": case.latent,
         "indexer": f"{case.H_i}x{case.D_i} {case.idx_dtype}", "top_k": case.K,
         "block_size": case.bs, "l2": L2_NOTE,
         "parallelism": f"replicas{world}" if world > 1 else "1gpu"}
    return c


def headline(args, world, res, peaks):
    """The JSON line of the measured workload from run_gpu's result: whole-job
    throughput (units of all ranks over the slowest rank's timed region), the
    dominant kernel's roofline and, for decode, the whole path's."""
    case = res["case"]
    units = (case.Nq if case.kind == "prefill" else case.B) * world
    value = units * args.steps / (res["total_ms"] / 1e3)
    roof, step_work = roofline_of(res, peaks)
    ms_step = res["total_ms"] / args.steps
    line = {
        "metric": metric_of(case), "value": value, "unit": unit_of(case), "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16+" + ("fp8" if case.idx_dtype == "fp8" else "bf16") + " (fp32 accumulate)",
        "data": "synthetic (seeded, shapes and distributions of the workload)",
        "config": config_of(case, world),
        "roofline": roof,
        "stage_ms": {"index_score": res["stage_ms"][0], "topk": res["stage_ms"][1],
                     "sparse_attn": res["stage_ms"][2]},
        "clocks": res["clocks"],
        "e2e": res["e2e"]["calls"] if res["e2e"] else None,
        "e2e_graph": res["e2e"]["graph"] if res["e2e"] else None,
        "e2e_step": res["e2e"].get("step") if res["e2e"] else None,
        "gpu_launches": res["launches"],
        "gpu_launches_per_step": res["launches_per"],
        "device_status": res["status"],
        "cache_write": res["cache_write"],
    }
    if res.get("step_calls") is not None:
        line["step_calls"] = res["step_calls"]
    if res.get("bounded_index") is not None:
        line["bounded_index"] = res["bounded_index"]
    line["path_roofline"] = path_roofline(case, ms_step, peaks)
    return line


def path_roofline(case, ms_step, peaks):
    """The whole step against its roofline: decode, the indexer keys plus the
    gathered rows over HBM bandwidth; prefill, the ideal time of its tensor
    work (FP8 indexer at twice the bf16 peak, bf16 attention) over the step."""
    alg = algorithmic(case)
    if case.kind == "decode":
        step_bytes = alg["index_bytes"] + alg["gather_bytes"]
        frac = step_bytes / (ms_step / 1e3) / 1e9 / peaks["hbm_gbs"]
        return {"bound": "hbm", "algorithmic_bytes_per_step": step_bytes, "frac": round(frac, 4),
                "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    ideal_s = (alg["index_flops"] / (peaks["bf16_tflops"] * 2e12) +
               alg["attn_flops"] / (peaks["bf16_tflops"] * 1e12))
    return {"bound": "tensor", "ideal_ms": round(ideal_s * 1e3, 4),
            "frac": round(ideal_s / (ms_step / 1e3), 4)}


def secondary_line(r2, st2, world, peaks):
    """One more workload measured in the same run (same timing rules)."""
    c2 = r2["case"]
    u2 = (c2.Nq if c2.kind == "prefill" else c2.B) * world
    roof2, _ = roofline_of(r2, peaks)
    ms2 = r2["total_ms"] / st2
    return {"metric": metric_of(c2), "value": u2 * st2 / (r2["total_ms"] / 1e3),
            "unit": unit_of(c2), "ms_per_step": ms2, "steps": st2,
            "config": config_of(c2, world), "roofline": roof2,
            "path_roofline": path_roofline(c2, ms2, peaks),
            "stage_ms": dict(zip(["index_score", "topk", "sparse_attn"], r2["stage_ms"])),
            "gpu_launches": r2["launches"], "gpu_launches_per_step": r2["launches_per"],
            "clocks": r2["clocks"], "device_status": r2["status"],
            "cache_write": r2["cache_write"], "step_calls": r2.get("step_calls"),
            "bounded_index": r2.get("bounded_index")}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="dec-batch",
                    choices=["dec-tiny", "dec-batch", "prefill", "long-dec", "million"])
    ap.add_argument("--secondary", default="prefill,dec-tiny,long-dec,million",
                    help="comma-separated extra workloads reported in the same line")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-step-seconds", type=float, default=4.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--prefill-tokens", type=int, default=None,
                    help="prompt length of the prefill workload (default 16384; smaller "
                         "prompts are for profiler captures, not bench lines)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    global PREFILL_TOKENS
    PREFILL_TOKENS = args.prefill_tokens

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        return run_reference(args, rank, world)

    import torch
    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")

    peaks = measured_peaks()
    res = run_gpu(args.workload, args.steps, args.warmup, rank, world, local_rank,
                  do_e2e=not args.no_e2e)
    case = res["case"]
    line = headline(args, world, res, peaks)
    extra = [w for w in args.secondary.split(",") if w and w != args.workload]
    for wname in extra:
        st2 = max(3, args.steps // 4)
        r2 = run_gpu(wname, st2, args.warmup, rank, world, local_rank, do_e2e=False)
        line[wname.replace("-", "_")] = secondary_line(r2, st2, world, peaks)
    if rank == 0 and world == 1:
        line["cpu_baseline"] = cpu_baseline(case, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
