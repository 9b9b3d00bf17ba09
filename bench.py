"""Benchmark of the paged q8-KV attention hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one pass of the whole hot path over one batch: kv_store of the
batch's new K/V rows (q8 quantize + scatter by slot) followed by
paged_attention over the cache (unified causal prefill/decode, split-KV
segments merged by LSE where the call splits).  The cache prefix is populated
before timing; inputs live in HBM when the timed region starts.

Headline workload: long-context decode at D = 256 (8 sequences x 131072 keys,
32 q / 8 kv heads, block size 16, 16 KV segments merged by LSE; 4.56 GB of
KV per step), the largest of the serving workloads that fits one GPU.  The
same run measures every serving workload (decode batch, chunked prefill,
mixed batch, long decode at D = 128 and 256) and reports each under
"workloads" with its own roofline fraction and clocks.
A workload whose KV bytes fit in twice the L2 gets a 512 MiB buffer write
between timed steps, outside the per-step CUDA events that time it.
Metric: algorithmic HBM bytes of a step / step time (GB/s); prefill-only
workloads report attention TFLOP/s instead.

Under torchrun (N > 1) every rank runs an independent replica (seed offset by
rank): the path has no exchange step, so there is no collective on the data
path; the ranks meet only at the timing barriers and the max-over-ranks.
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
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_attention_int8_gb300 import _lib, build as pkg_build, inputs  # noqa: E402

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_BYTES = 129e6
FLUSH_BYTES = 512 << 20  # written between timed steps when the working set fits in L2


# ----------------------------------------------------------------------------- work accounting

def step_work(w: inputs.Workload) -> dict:
    """Algorithmic bytes and FLOPs of one step (see the design notes).

    attention: every visible (row, key) pair's K and V codes + fp16 scales
    once per kv head (sum_s L_s * Hk * 2 * (D + 2 * D/32)), plus q read, out and
    lse written, the block-table entries used and the metadata;
    kv_store: N * Hk * (4D read + 2(D + D/16) written) for the N rows with a
    slot, + 8 slot bytes for every row (padding rows, slot < 0, are only
    looked up)."""
    s = w.spec
    G = s.d // 32
    L = w.seq_lens.to(torch.int64)
    T, S = w.num_tokens, w.num_seqs
    kv = int(L.sum()) * s.hk * 2 * (s.d + 2 * G)
    q_out = T * s.hq * s.d * 2 * 2 + T * s.hq * 4
    pages = int(((L + s.bs - 1) // s.bs).sum()) * 4
    meta = (2 * S + 1) * 4
    attn_bytes = kv + q_out + pages + meta
    n_rows = int(w.new_slots.shape[0])
    n_new = int((w.new_slots >= 0).sum())
    store_bytes = n_new * s.hk * (4 * s.d + 2 * (s.d + 2 * G)) + 8 * n_rows
    # visible (row, key) pairs: token i of sequence s sees ctx + i + 1 keys
    ql = w.q_lens.to(torch.int64)
    ctx = L - ql
    pairs = int((ql * ctx + ql * (ql + 1) // 2).sum()) * s.hq
    flops = 4 * s.d * pairs
    return dict(attn_bytes=attn_bytes, store_bytes=store_bytes, step_bytes=attn_bytes + store_bytes,
                kv_bytes=kv, flops=flops, pairs=pairs)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


# The sources of the kernels one paged_attention call launches (their host
# dispatch included); a recorded ncu figure holds while these are unchanged.
ATTENTION_SOURCES = ("attention.cu", "attn_decode.cu", "attn_prefill.cu", "attn_prefill_tc.cu",
                     "attn_common.cuh", "attn_f8v4.cuh", "common.cuh", "tcgen05.cuh", "launch.h")


def kernel_sources_sha256() -> str:
    """One hash over the attention kernels' source files (any change
    invalidates a recorded ncu figure)."""
    d = os.path.join(ROOT, "paged_attention_int8_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(ATTENTION_SOURCES):
        h.update(name.encode())
        h.update(open(os.path.join(d, name), "rb").read())
    return h.hexdigest()


def recorded_traffic(workload: str):
    """Per-call DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum over
    the kernels of one paged_attention call) from the committed ncu summary
    profiles/attention_<workload>.md, if it was taken on the current kernel
    sources; else None."""
    path = os.path.join(ROOT, "profiles", f"attention_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    rec_sha, traffic = None, None
    for line in text.splitlines():
        if line.startswith("source_sha256:"):
            rec_sha = line.split(":", 1)[1].strip()
        if line.startswith("traffic_bytes_per_launch:"):
            traffic = float(line.split(":", 1)[1].strip())
    return traffic if rec_sha == kernel_sources_sha256() else None


def attention_launches(spec: inputs.Spec, max_query_len: int, num_splits: int) -> int:
    """Kernels one paged_attention call launches (the dispatch rule of the
    library): the decode kernel when a kv head stacks at most 8 q heads, a
    prefill kernel when some sequence has several query tokens (or the heads
    do not fit the decode kernel), the segment reduce when splitting."""
    use_decode = spec.hq // spec.hk <= 8
    use_prefill = (not use_decode) or max_query_len > 1
    return int(use_decode) + int(use_prefill) + int(num_splits > 1)


# ----------------------------------------------------------------------------- replicas

def replica_spec(spec: inputs.Spec, rank: int) -> inputs.Spec:
    """Rank r runs the same workload shape with its own seed (independent
    replicas: the path has no exchange step)."""
    return spec.replace(seed=spec.seed + 1000 * rank) if rank else spec


def reduce_over_ranks(ms_total: float, units: float, device) -> tuple:
    """(slowest rank's time, units all ranks processed): the whole-job
    throughput is the second over the first."""
    import torch.distributed as dist
    t = torch.tensor([ms_total], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    u = torch.tensor([units], dtype=torch.float64, device=device)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (SM clock, throttle reasons) while the timed region runs."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, t0: float, t1: float):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = [l.split(", ") for (ts, l) in self.lines if t0 - 0.05 <= ts <= t1 + 0.05]
        if not rows:
            rows = [l.split(", ") for (_, l) in self.lines[-3:]]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[2]))
                mx.append(float(r[3]))
                for n, v in zip(names, r[6:10]):
                    if v.strip() == "Active":
                        reasons.add(n)
            except (IndexError, ValueError):
                continue
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- GPU arm

class Runner:
    def __init__(self, w: inputs.Workload, device, num_splits=None):
        s = w.spec
        self.w, self.device = w, device
        self.kc, self.ks, self.vc, self.vs = inputs.empty_cache(w.num_blocks, s.hk, s.bs, s.d,
                                                                device=device, canary=False)
        self.status = torch.zeros(4, dtype=torch.int32, device=device)
        # populate the cached prefix (untimed)
        if w.prefix_key.shape[0]:
            chunk = 1 << 18
            for a in range(0, w.prefix_key.shape[0], chunk):
                _lib.kv_store(w.prefix_key[a:a + chunk].to(device),
                              w.prefix_value[a:a + chunk].to(device),
                              w.prefix_slots[a:a + chunk].to(device),
                              self.kc, self.ks, self.vc, self.vs, status=self.status)
        self.new_k = w.new_key.to(device)
        self.new_v = w.new_value.to(device)
        self.slots = w.new_slots.to(device)
        self.q = w.q.to(device)
        self.cu = w.cu_seqlens_q.to(device)
        self.seq_lens = w.seq_lens.to(device)
        self.bt = w.block_table.to(device)
        self.ns = s.num_splits if num_splits is None else num_splits
        self.ns_eff = self.ns or _lib.auto_num_splits(w.num_seqs, s.hk, w.max_query_len,
                                                      w.max_seq_len)
        self.ws = torch.zeros(_lib.workspace_size(w.num_seqs, s.hq, s.d, self.ns_eff),
                              dtype=torch.uint8, device=device)
        self.out = torch.empty_like(self.q)
        self.lse = torch.empty((w.num_tokens, s.hq), dtype=torch.float32, device=device)
        self.launches_per_step = 1 + attention_launches(s, w.max_query_len, self.ns_eff)

    def step(self, ev=None):
        w = self.w
        _lib.kv_store(self.new_k, self.new_v, self.slots, self.kc, self.ks, self.vc, self.vs,
                      status=self.status)
        if ev is not None:
            ev[0].record()
        _lib.paged_attention(self.q, self.kc, self.ks, self.vc, self.vs, self.cu, self.seq_lens,
                             self.bt, w.max_query_len, w.max_seq_len, w.softmax_scale,
                             num_splits=self.ns_eff, out=self.out, lse=self.lse,
                             workspace=self.ws)
        if ev is not None:
            ev[1].record()

    def check(self):
        torch.cuda.synchronize()
        assert _lib.check_status(self.status) == 0
        assert _lib.check_status(self.ws) == 0


def kv_store_measure(r: Runner, reps: int = 20):
    """kv_store alone on the workload's prefix rows (the cache population
    batch; storing the same rows again is idempotent): algorithmic bytes
    (bf16 K/V read, codes + scales written, slots read) per CUDA-event time."""
    w = r.w
    s = w.spec
    n = int(w.prefix_slots.shape[0])
    if n == 0:
        return None
    G = s.d // 32
    k, v, sl = (w.prefix_key.to(r.device), w.prefix_value.to(r.device),
                w.prefix_slots.to(r.device))
    nbytes = n * s.hk * (4 * s.d + 2 * (s.d + 2 * G)) + 8 * n
    for _ in range(3):
        _lib.kv_store(k, v, sl, r.kc, r.ks, r.vc, r.vs, status=r.status)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(reps)]
    for a, b in ev:
        a.record()
        _lib.kv_store(k, v, sl, r.kc, r.ks, r.vc, r.vs, status=r.status)
        b.record()
    torch.cuda.synchronize()
    assert _lib.check_status(r.status) == 0
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    del k, v, sl
    return {"tokens": n, "bytes": nbytes, "ms": round(ms, 5),
            "achieved_gbs": round(nbytes / (ms * 1e-3) * 1e-9, 2)}


def norm_rope_measure(r: Runner, reps: int = 20):
    """kv_store_norm_rope alone on the workload's prefix rows (the cache
    population batch, stored again): each key row through a weighted RMSNorm
    and a full rotary embedding (positions = the tokens' places in their
    sequences, the usual rotary frequencies) before q8, values as kv_store.
    Algorithmic bytes: bf16 K/V read, codes and scales written, slots and
    positions read, each token's cos/sin row and the norm weight once."""
    w = r.w
    s = w.spec
    n = int(w.prefix_slots.shape[0])
    if n == 0:
        return None
    L = w.seq_lens.to(torch.int64)
    ctx = L - w.q_lens.to(torch.int64)
    pos = torch.cat([torch.arange(int(c), dtype=torch.int64) for c in ctx.tolist()])
    max_pos = int(ctx.max().item()) if ctx.numel() else 1
    pairs = s.d // 2
    inv_freq = 10000.0 ** (-torch.arange(pairs, dtype=torch.float64) / pairs)
    ang = torch.arange(max(max_pos, 1), dtype=torch.float64)[:, None] * inv_freq[None, :]
    table = torch.stack([ang.cos(), ang.sin()], -1).to(torch.float32).to(r.device)
    wt = (torch.rand(s.d, generator=torch.Generator().manual_seed(5)) + 0.5).to(
        torch.bfloat16).to(r.device)
    k, v, sl = (w.prefix_key.to(r.device), w.prefix_value.to(r.device),
                w.prefix_slots.to(r.device))
    pos = pos.to(r.device)

    def call():
        _lib.kv_store_norm_rope(k, v, sl, r.kc, r.ks, r.vc, r.vs, positions=pos, norm_weight=wt,
                                rope=table, status=r.status)

    for _ in range(3):
        call()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(reps)]
    for a, b in ev:
        a.record()
        call()
        b.record()
    torch.cuda.synchronize()
    assert _lib.check_status(r.status) == 0
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    G = s.d // 32
    nbytes = n * (s.hk * (4 * s.d + 2 * (s.d + 2 * G)) + 4 * s.d + 16) + 2 * s.d
    del k, v, sl, pos, table, wt
    return {"tokens": n, "bytes": nbytes, "ms": round(ms, 5),
            "achieved_gbs": round(nbytes / (ms * 1e-3) * 1e-9, 2),
            "rotary_dim": s.d, "norm": True}


def options_measure(r: Runner, unit: str, reps: int = 20, window: int = 1024):
    """The attention options on the workload's own batch, timed with CUDA
    events: for a decode batch a sliding window of `window` keys with a sink
    logit per q head (algorithmic bytes: the visible keys' K/V codes and
    scales, q, out, lse, the visible pages' block-table entries, the sinks);
    for a prefill batch the non-causal prefix pass, every query over all of
    its sequence's keys (FLOPs: 4 D per (row, key) pair)."""
    w = r.w
    s = w.spec
    G = s.d // 32
    L = w.seq_lens.to(torch.int64)
    ql = w.q_lens.to(torch.int64)
    T = w.num_tokens
    out = torch.empty_like(r.q)
    lse = torch.empty((T, s.hq), dtype=torch.float32, device=r.device)
    ws = torch.zeros_like(r.ws)
    ns = r.ns_eff
    if unit == "TFLOP/s":
        kw = dict(causal=False)
        flops = 4 * s.d * s.hq * int((ql * L).sum())
    else:
        sinks = (torch.rand(s.hq, generator=torch.Generator().manual_seed(9)) * 4.0 - 1.0).to(
            r.device)
        kw = dict(sinks=sinks, sliding_window=window)
        ns = 0  # the library's automatic split count, sized for the window
        vis = torch.clamp(L, max=window)
        nbytes = (int(vis.sum()) * s.hk * 2 * (s.d + 2 * G) + T * s.hq * (4 * s.d + 4)
                  + int(((vis + s.bs - 1) // s.bs + 1).sum()) * 4 + (2 * w.num_seqs + 1) * 4
                  + s.hq * 4)

    def call():
        _lib.paged_attention(r.q, r.kc, r.ks, r.vc, r.vs, r.cu, r.seq_lens, r.bt, w.max_query_len,
                             w.max_seq_len, w.softmax_scale, num_splits=ns, out=out,
                             lse=lse, workspace=ws, **kw)

    for _ in range(3):
        call()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(reps)]
    for a, b in ev:
        a.record()
        call()
        b.record()
    torch.cuda.synchronize()
    assert _lib.check_status(ws) == 0
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    hbm_peak, tc_peak, _ = load_peaks()
    if unit == "TFLOP/s":
        tf = flops / (ms * 1e-3) * 1e-12
        return {"option": "non-causal prefix pass", "flops": flops, "ms": round(ms, 5),
                "tflops": round(tf, 2), "peak": tc_peak, "frac": round(tf / tc_peak, 4)}
    gbs = nbytes / (ms * 1e-3) * 1e-9
    return {"option": f"sliding window {window} + sinks", "bytes": nbytes, "ms": round(ms, 5),
            "achieved_gbs": round(gbs, 2), "peak": hbm_peak, "frac": round(gbs / hbm_peak, 4)}


MERGE_ROWS = 1 << 19  # (token, q head) rows of the merge measurement


def merge_measure(r: Runner, reps: int = 20):
    """merge_attn_states of two attention states over MERGE_ROWS (token, q
    head) rows of the workload's head size -- a cached-prefix pass and a
    new-key pass of a large prefill batch, seeded synthetic values (the
    step's own output is too small to measure bandwidth on): algorithmic
    bytes (two bf16 outputs and two LSEs read, the merged output and LSE
    written) per CUDA-event time."""
    d = r.out.shape[-1]
    rows = MERGE_ROWS
    gen = torch.Generator(device=r.device).manual_seed(7)
    out_a = torch.randn((rows, 1, d), generator=gen, device=r.device).to(torch.bfloat16)
    out_b = torch.randn((rows, 1, d), generator=gen, device=r.device).to(torch.bfloat16)
    lse_a = torch.randn((rows, 1), generator=gen, device=r.device) * 4.0
    lse_b = torch.randn((rows, 1), generator=gen, device=r.device) * 4.0
    merged = torch.empty_like(out_a)
    lse_m = torch.empty_like(lse_a)
    nbytes = rows * (3 * d * 2 + 3 * 4)

    def call():
        _lib.merge_attn_states(out_a, lse_a, out_b, lse_b, out=merged, lse=lse_m)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(3):
            call()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    try:
        # the calls replayed from a CUDA graph: device time, no host launch cost
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(reps):
                call()
        graph.replay()
        torch.cuda.synchronize()
        a.record()
        graph.replay()
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / reps
        timing = f"CUDA graph of {reps} calls, replayed"
        del graph
    except RuntimeError:
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(reps)]
        for a, b in ev:
            a.record()
            call()
            b.record()
        torch.cuda.synchronize()
        ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
        timing = "CUDA events around each call"
    del out_a, out_b, lse_b, lse_a, merged, lse_m
    return {"rows": rows, "bytes": nbytes, "ms": round(ms, 5),
            "achieved_gbs": round(nbytes / (ms * 1e-3) * 1e-9, 2), "timing": timing,
            "l2": "inputs larger than L2" if rows * (4 * d + 8) > L2_BYTES else "inputs fit in L2"}


def f8v4_measure(w: inputs.Workload, device, flops=None, reps: int = 20):
    """The same batch stored in the fp8 / 4-bit format (e4m3 keys, 4-bit
    values with a per-key fp16 scale and zero) and attended by
    paged_attention_f8v4.  Decode batches: algorithmic bytes per call (D +
    D/2 + 4 per visible (key, kv head), q, out, lse, block-table entries,
    metadata) per CUDA-event time; prefill batches (``flops`` given): FLOPs
    per CUDA-event time against the tensor peak."""
    s = w.spec
    kc, vc, vs, vz = inputs.empty_cache_f8v4(w.num_blocks, s.hk, s.bs, s.d, device=device,
                                             canary=False)
    k, v, sl = w.all_key_value()
    chunk = 1 << 18
    for a in range(0, k.shape[0], chunk):
        _lib.kv_store_f8v4(k[a:a + chunk].to(device), v[a:a + chunk].to(device),
                           sl[a:a + chunk].to(device), kc, vc, vs, vz)
    # the store alone on the population batch (the prefix rows, stored again:
    # idempotent): bf16 K/V read, codes, nibbles, scales and zeros written
    pk, pv, ps = (w.prefix_key.to(device), w.prefix_value.to(device),
                  w.prefix_slots.to(device))
    n = int(ps.shape[0])
    store = None
    if n:
        for _ in range(3):
            _lib.kv_store_f8v4(pk, pv, ps, kc, vc, vs, vz)
        sev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(reps)]
        for a, b in sev:
            a.record()
            _lib.kv_store_f8v4(pk, pv, ps, kc, vc, vs, vz)
            b.record()
        torch.cuda.synchronize()
        sms = statistics.mean(a.elapsed_time(b) for a, b in sev)
        sbytes = n * s.hk * (4 * s.d + s.d + s.d // 2 + 4) + 8 * n
        store = {"tokens": n, "bytes": sbytes, "ms": round(sms, 5),
                 "achieved_gbs": round(sbytes / (sms * 1e-3) * 1e-9, 2)}
    del pk, pv, ps
    q, cu = w.q.to(device), w.cu_seqlens_q.to(device)
    seq_lens, bt = w.seq_lens.to(device), w.block_table.to(device)
    ns = _lib.auto_num_splits(w.num_seqs, s.hk, w.max_query_len, w.max_seq_len)
    ws = torch.zeros(_lib.workspace_size(w.num_seqs, s.hq, s.d, ns), dtype=torch.uint8,
                     device=device)
    out = torch.empty_like(q)
    lse = torch.empty((w.num_tokens, s.hq), dtype=torch.float32, device=device)

    def call():
        _lib.paged_attention_f8v4(q, kc, vc, vs, vz, cu, seq_lens, bt, w.max_query_len,
                                  w.max_seq_len, w.softmax_scale, num_splits=ns, out=out, lse=lse,
                                  workspace=ws)

    for _ in range(3):
        call()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(reps)]
    for a, b in ev:
        a.record()
        call()
        b.record()
    torch.cuda.synchronize()
    assert _lib.check_status(ws) == 0
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    L = w.seq_lens.to(torch.int64)
    kv = int(L.sum()) * s.hk * (s.d + s.d // 2 + 4)
    T = w.num_tokens
    nbytes = kv + T * s.hq * s.d * 4 + T * s.hq * 4 + int(((L + s.bs - 1) // s.bs).sum()) * 4 \
        + (2 * w.num_seqs + 1) * 4
    hbm_peak, tc_peak, _ = load_peaks()
    gbs = nbytes / (ms * 1e-3) * 1e-9
    del kc, vc, vs, vz, ws
    if store is not None:
        store["peak"] = hbm_peak
        store["frac"] = round(store["achieved_gbs"] / hbm_peak, 4)
    res = {"format": "fp8 e4m3 keys, 4-bit values with fp16 scale and zero per key",
           "bytes": nbytes, "ms": round(ms, 5), "achieved_gbs": round(gbs, 2),
           "num_splits": ns, "kv_store_f8v4": store}
    if flops is None:
        res.update(peak=hbm_peak, frac=round(gbs / hbm_peak, 4))
    else:
        tf = flops / (ms * 1e-3) * 1e-12
        res.update(flops=flops, tflops=round(tf, 2), peak=tc_peak, frac=round(tf / tc_peak, 4))
    return res


def e2e_measure(r: Runner, steps: int, warmup: int):
    """Same step through the public API with the step's inputs copied from
    pinned host memory and the outputs read back, all inside the timed region."""
    w = r.w
    host_in = [t.pin_memory() for t in (w.q, w.new_key, w.new_value, w.new_slots,
                                        w.cu_seqlens_q, w.seq_lens, w.block_table)]
    dev_in = [r.q, r.new_k, r.new_v, r.slots, r.cu, r.seq_lens, r.bt]
    host_out = torch.empty(r.out.shape, dtype=r.out.dtype).pin_memory()
    host_lse = torch.empty(r.lse.shape, dtype=r.lse.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = host_out.numel() * 2 + host_lse.numel() * 4

    def one():
        for h, d in zip(host_in, dev_in):
            d.copy_(h, non_blocking=True)
        r.step()
        host_out.copy_(r.out, non_blocking=True)
        host_lse.copy_(r.lse, non_blocking=True)

    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        one()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps, h2d, d2h


# ----------------------------------------------------------------------------- oracle arm

def oracle_state(w: inputs.Workload):
    import oracle
    s = w.spec
    kc, ks, vc, vs = [t.numpy() for t in inputs.empty_cache(w.num_blocks, s.hk, s.bs, s.d,
                                                            canary=False)]
    ks, vs = ks.view(np.uint16), vs.view(np.uint16)
    if w.prefix_key.shape[0]:
        oracle.kv_store(inputs.bf16_bits(w.prefix_key), inputs.bf16_bits(w.prefix_value),
                        w.prefix_slots.numpy(), kc, ks, vc, vs)
    return kc, ks, vc, vs


def oracle_sample_step(w, caches, rows, threads):
    """The oracle's pass over one sample: kv_store of the new rows, then
    attention for the sampled (token, head) rows."""
    import oracle
    kc, ks, vc, vs = caches
    oracle.kv_store(inputs.bf16_bits(w.new_key), inputs.bf16_bits(w.new_value),
                    w.new_slots.numpy(), kc, ks, vc, vs, n_threads=threads)
    oracle.paged_attention(inputs.bf16_bits(w.q), kc, ks, vc, vs, w.cu_seqlens_q.numpy(),
                           w.seq_lens.numpy(), w.block_table.numpy(), w.softmax_scale,
                           rows=rows, n_threads=threads)


def sample_bytes(w, rows) -> float:
    """Algorithmic bytes of the sampled rows: their KV bytes (per q head,
    i.e. a share 1/qpk of the kv head's stream) plus q/out/lse."""
    s = w.spec
    G = s.d // 32
    cu = w.cu_seqlens_q.numpy()
    L = w.seq_lens.numpy()
    ql = w.q_lens.numpy()
    tok = rows // s.hq
    seq = np.searchsorted(cu, tok, side="right") - 1
    keys = (L[seq] - ql[seq]) + (tok - cu[seq]) + 1
    qpk = s.hq // s.hk
    kv = float(np.sum(L[seq] / ql[seq].clip(min=1))) * 2 * (s.d + 2 * G) / qpk
    return kv + rows.shape[0] * (s.d * 4 + 4), float(np.sum(keys)) * 4 * s.d


def cpu_baseline(w, budget_s: float = 20.0):
    threads = os.cpu_count() or 1
    caches = oracle_state(w)
    rows_all = np.arange(w.num_tokens * w.spec.hq, dtype=np.int64)
    rng = np.random.default_rng(0)
    # calibrate on a small sample, then size the sample to the budget
    probe = np.sort(rng.choice(rows_all, size=min(rows_all.size, 4 * threads), replace=False))
    t0 = time.perf_counter()
    oracle_sample_step(w, caches, probe, threads)
    per_row = (time.perf_counter() - t0) / probe.size
    n = int(min(rows_all.size, max(probe.size, budget_s / max(per_row, 1e-9))))
    rows = np.sort(rng.choice(rows_all, size=n, replace=False))
    t0 = time.perf_counter()
    oracle_sample_step(w, caches, rows, threads)
    dt = time.perf_counter() - t0
    b, f = sample_bytes(w, rows)
    store = step_work(w)["store_bytes"]
    return {"bytes": b + store, "flops": f, "seconds": dt, "rows": int(n),
            "rows_total": int(rows_all.size), "cores": threads}


# ----------------------------------------------------------------------------- main

METRIC = "paged q8-KV attention: decode HBM GB/s (% of peak), prefill TFLOP/s"


def metric_for(spec: inputs.Spec):
    """Prefill-only workloads are tensor-bound (TFLOP/s); the rest HBM-bound (GB/s)."""
    if spec.n_prefill and not spec.n_decode and not spec.fixed_decode_lens:
        return METRIC, "TFLOP/s", "tensor"
    return METRIC, "GB/s", "hbm"


# The default line: the largest workload that fits one GPU (4.56 GB of KV per
# step), with every serving workload measured in the same process beside it.
HEADLINE = "long_decode_d256"
SUITE = ("decode_batch", "chunked_prefill", "mixed_batch", "long_decode", "long_decode_d256")


def timed_steps(r: Runner, steps: int, flush: bool, world: int, device):
    """Time exactly `steps` steps between barriers and synchronizes, sampling
    the SM clocks meanwhile.  Returns (ms of all steps, mean ms of the
    attention call alone, clocks)."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    flush_buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device) if flush else None
    steps_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(steps)] if flush else None
    clocks = ClockSampler(device.index)
    clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    e0.record()
    for i in range(steps):
        if flush:
            # a working set that fits in L2 would be served from it on the
            # next step: write a buffer larger than L2 between timed steps,
            # outside the per-step events
            flush_buf.fill_(i & 0xFF)
            steps_ev[i][0].record()
        r.step(ev[i])
        if flush:
            steps_ev[i][1].record()
    e1.record()
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    clk = clocks.stop(t_wall0, t_wall1)
    if flush:
        ms_total = sum(a.elapsed_time(b) for a, b in steps_ev)
    else:
        ms_total = e0.elapsed_time(e1)
    attn_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    del flush_buf
    return ms_total, attn_ms, clk


def roofline_of(name, spec, w, work, attn_ms, ns_eff, hbm_peak, tc_peak, peak_src):
    """Roofline of the attention call (the dominant kernels of a step).

    HBM-bound workloads: algorithmic bytes per call / call time against the
    measured copy bandwidth.  Prefill: attention FLOPs / call time against the
    measured dense bf16 peak.  A batch with both (the mixed batch) also gets
    both parts, bytes / bandwidth and FLOPs / peak, and the larger of the two
    as the roofline time."""
    _, _, bound = metric_for(spec)
    bytes_ms = work["attn_bytes"] / (hbm_peak * 1e9) * 1e3
    flops_ms = work["flops"] / (tc_peak * 1e12) * 1e3
    if bound == "hbm":
        achieved = work["attn_bytes"] / (attn_ms * 1e-3) * 1e-9
        peak, runit = hbm_peak, "GB/s"
    else:
        achieved = work["flops"] / (attn_ms * 1e-3) * 1e-12
        peak, runit = tc_peak, "TFLOP/s"
    traffic = recorded_traffic(name)
    roof = {"bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": runit,
            "frac": round(achieved / peak, 4), "traffic": traffic,
            "traffic_source": (f"profiles/attention_{name}.md (ncu dram bytes, recorded on the "
                               "current kernel sources)") if traffic is not None else None,
            "kernel": "paged_attention call (%d kernel launches)"
                      % attention_launches(spec, w.max_query_len, ns_eff),
            "launch_ms": round(attn_ms, 5), "peak_source": peak_src,
            "algorithmic_per_launch": work["attn_bytes"] if bound == "hbm" else work["flops"]}
    if spec.n_prefill and (spec.n_decode or spec.fixed_decode_lens):
        roof["parts"] = {"bytes_ms": round(bytes_ms, 6), "flops_ms": round(flops_ms, 6),
                         "roofline_ms": round(max(bytes_ms, flops_ms), 6),
                         "frac_of_roofline_time": round(max(bytes_ms, flops_ms) / attn_ms, 4),
                         "tflops": round(work["flops"] / (attn_ms * 1e-3) * 1e-12, 2)}
    return roof


def run_workload(name, args, device, rank, world, headline: bool):
    """Build one workload, time it, and measure its extras.  Returns the
    entry of the JSON line (and the headline's fields when asked)."""
    spec = inputs.WORKLOADS[name]
    metric, unit, bound = metric_for(spec)
    w = inputs.make_workload(replica_spec(spec, rank))
    work = step_work(w)
    r = Runner(w, device, args.num_splits)
    for _ in range(args.warmup):
        r.step()
    r.check()
    flush = work["kv_bytes"] <= 2 * L2_BYTES
    ms_total, attn_ms, clk = timed_steps(r, args.steps, flush, world, device)
    r.check()
    units_local = work["flops"] if unit == "TFLOP/s" else work["step_bytes"]
    if world > 1:
        ms_total, units_per_step = reduce_over_ranks(ms_total, units_local, device)
    else:
        units_per_step = units_local
    ms_step = ms_total / args.steps
    scale = 1e-12 if unit == "TFLOP/s" else 1e-9
    value = units_per_step / (ms_step * 1e-3) * scale
    hbm_peak, tc_peak, peak_src = load_peaks()
    entry = {"value": round(value, 3), "unit": unit, "ms_per_step": round(ms_step, 5),
             "roofline": roofline_of(name, spec, w, work, attn_ms, r.ns_eff, hbm_peak, tc_peak,
                                     peak_src),
             "clocks": clk,
             "config": {"workload": name, "num_seqs": w.num_seqs, "num_tokens": w.num_tokens,
                        "q_heads": spec.hq, "kv_heads": spec.hk, "head_dim": spec.d,
                        "block_size": spec.bs, "max_seq_len": w.max_seq_len,
                        "sum_kv_len": int(w.seq_lens.sum()), "num_splits": r.ns_eff,
                        "l2": ("L2 flushed between steps (%d MiB written, untimed)"
                               % (FLUSH_BYTES >> 20)) if flush
                        else "inputs larger than L2 (no flush)"},
             "step_bytes": work["step_bytes"], "step_flops": work["flops"],
             "gpu_launches": r.launches_per_step * args.steps}
    if rank == 0 and not args.no_kv_store:
        store = kv_store_measure(r)
        if store is not None:
            store["peak"] = hbm_peak
            store["frac"] = round(store["achieved_gbs"] / hbm_peak, 4)
        entry["kv_store"] = store
    if rank == 0 and name in ("decode_batch", "chunked_prefill") and not args.no_kv_store:
        entry["options"] = options_measure(r, unit)
    if rank == 0 and name == "decode_batch" and not args.no_kv_store:
        # the fused norm + rotation store on the same population batch
        nr = norm_rope_measure(r)
        if nr is not None:
            hbm_peak_nr, _, _ = load_peaks()
            nr["peak"] = hbm_peak_nr
            nr["frac"] = round(nr["achieved_gbs"] / hbm_peak_nr, 4)
        entry["kv_store_norm_rope"] = nr
    if rank == 0 and name in ("decode_batch", "chunked_prefill") and not args.no_kv_store:
        # the alternative format on the same batch: fewer bytes per key
        f8 = f8v4_measure(w, device, flops=work["flops"] if unit == "TFLOP/s" else None)
        f8["vs_q8_call"] = round(f8["ms"] / attn_ms, 4)
        entry["f8v4"] = f8
    if headline and rank == 0:
        if not args.no_kv_store:
            merge = merge_measure(r)
            merge["peak"] = hbm_peak
            merge["frac"] = round(merge["achieved_gbs"] / hbm_peak, 4)
            entry["merge_attn_states"] = merge
        if not args.no_e2e:
            e2e_ms, h2d, d2h = e2e_measure(r, max(10, args.steps // 10), 5)
            entry["e2e"] = {"value": units_local / (e2e_ms * 1e-3) * scale, "unit": unit,
                            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                            "ms_per_step": e2e_ms}
        if world == 1 and not args.no_cpu_baseline:
            cb = cpu_baseline(w)
            cv = (cb["flops"] * 1e-12 if unit == "TFLOP/s" else cb["bytes"] * 1e-9) / cb["seconds"]
            entry["cpu_baseline"] = {
                "value": round(cv, 4), "unit": unit, "cores": cb["cores"], "kind": "oracle",
                "sample": f"kv_store of the step's {int(w.new_slots.shape[0])} new rows + "
                          f"fp64 attention of {cb['rows']} of {cb['rows_total']} (token, q head) "
                          f"rows, {cb['seconds']:.1f} s"}
    del r, w
    torch.cuda.empty_cache()
    return entry


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(inputs.WORKLOADS),
                    help="the workload of the line's headline value")
    ap.add_argument("--only", action="store_true",
                    help="measure the headline workload alone (no 'workloads' suite)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--num-splits", type=int, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-kv-store", action="store_true",
                    help="skip the separate kv_store and merge_attn_states throughput measurements")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    spec = inputs.WORKLOADS[args.workload]
    metric, unit, bound = metric_for(spec)

    if args.impl == "reference":
        run_reference(args, spec, metric, unit, world, rank)
        return

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    if rank == 0:
        pkg_build.build()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()

    suite = {}
    if not args.only:
        for name in SUITE:
            if name != args.workload:
                suite[name] = run_workload(name, args, device, rank, world, headline=False)
    head = run_workload(args.workload, args, device, rank, world, headline=True)
    suite[args.workload] = {k: v for k, v in head.items()
                            if k not in ("e2e", "cpu_baseline", "merge_attn_states")}

    if rank == 0:
        line = {
            "metric": metric, "value": head["value"], "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "int8 cache, fp16 mma, fp32 softmax", "data": "synthetic",
            "config": dict(head["config"], parallelism=f"replicas x{world}"),
            "roofline": head["roofline"], "kv_store": head.get("kv_store"),
            "merge_attn_states": head.get("merge_attn_states"),
            "cpu_baseline": head.get("cpu_baseline"), "e2e": head.get("e2e"),
            "gpu_launches": sum(e["gpu_launches"] for e in suite.values()),
            "clocks": head["clocks"],
            "step_bytes": head["step_bytes"], "step_flops": head["step_flops"],
            "workloads": {n: suite[n] for n in SUITE if n in suite},
        }
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_reference(args, spec, metric, unit, world, rank):
    """The oracle as the reference arm: each step one bounded sample of the
    workload on the host cores, sized so that warmup + steps fit ~2 minutes."""
    if rank != 0:
        return
    w = inputs.make_workload(spec)
    threads = os.cpu_count() or 1
    caches = oracle_state(w)
    rows_all = np.arange(w.num_tokens * spec.hq, dtype=np.int64)
    rng = np.random.default_rng(0)
    probe = np.sort(rng.choice(rows_all, size=min(rows_all.size, 2 * threads), replace=False))
    t0 = time.perf_counter()
    oracle_sample_step(w, caches, probe, threads)
    per_row = (time.perf_counter() - t0) / probe.size
    budget = 120.0 / (args.steps + args.warmup)
    n = int(min(rows_all.size, max(1, budget / max(per_row, 1e-9))))
    rows = np.sort(rng.choice(rows_all, size=n, replace=False))
    for _ in range(args.warmup):
        oracle_sample_step(w, caches, rows, threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_sample_step(w, caches, rows, threads)
    dt = (time.perf_counter() - t0) / args.steps
    b, f = sample_bytes(w, rows)
    b += step_work(w)["store_bytes"]
    value = (f * 1e-12 if unit == "TFLOP/s" else b * 1e-9) / dt
    line = {"impl": "reference", "metric": metric, "value": round(value, 5), "unit": unit,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "num_seqs": w.num_seqs,
                       "num_tokens": w.num_tokens, "q_heads": spec.hq, "kv_heads": spec.hk,
                       "head_dim": spec.d, "block_size": spec.bs, "max_seq_len": w.max_seq_len,
                       "sum_kv_len": int(w.seq_lens.sum()),
                       "parallelism": f"replicas x{world}"},
            "cpu_baseline": {"value": round(value, 5), "unit": unit, "cores": threads,
                             "kind": "oracle",
                             "sample": f"{n} of {rows_all.size} (token, q head) rows per step"},
            "e2e": {"value": round(value, 5), "unit": unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


if __name__ == "__main__":
    main()
