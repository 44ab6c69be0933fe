#!/usr/bin/env python
"""Benchmark of the INT4 per-token-head KV cache hot path on GB300.

A step is one pass of the whole hot path over one batch of synthetic input:
write the step's new K/V (randomized Hadamard rotation, bf16 rounding,
absmax scale, INT4 pack, slot scatter) and then paged attention over the
INT4 cache (query rotation, dequantised tiles, online softmax, split-KV
reduce, inverse rotation).  The default workload is the long-context decode
batch (Llama-3-8B shape: 32 q / 8 kv heads, head 128, block 16, 256
sequences x 32768 keys, a 9.1 GB cache, larger than L2, so no flush is
needed between steps).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

prints one JSON line.  With N > 1 every rank runs its own replica of the
workload (weak scaling, no collective on the data path); the timed region is
bracketed by a barrier and synchronize on every rank and the slowest rank's
time is used.  Launched without torchrun, `--gpus N` re-runs this script
under torch.distributed.run with N ranks on this node.

--impl reference times the fp64 CPU oracle on the host cores (rank 0 only)
on a bounded sample of the same workload: one process per host core, and in
each step every process does one unit step, the oracle's write of one new
token plus its attention for one (sequence, kv head) unit of the batch (a
unit is 1/num_kv_heads of a decode token).  The CPU baseline of our arm is
the same runner for --cpu-seconds.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "INT4-KV paged decode: KV-read GB/s vs HBM peak, tokens/s; RHT+quant write GB/s"
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_TC_TFLOPS = 1700.0  # dense bf16, sustained, one earlier GB300 measurement
WORKLOAD_TEXT = {
    "tiny": "tiny causal: 4 q / 4 kv heads, head 128, block 16, seqs (q,kv) = (4,128),(4,97)",
    "phi3": "Phi-3-mini decode: 32 q / 32 kv heads, head 96 (b=32, n=3), block 16, batch 32 x kv 1024, 1% outlier channels x8",
    "gqa": "Llama-3.2-1B GQA decode: 32 q / 8 kv heads, head 128, block 16, batch 64, kv ~ U[512, 8192]",
    "mixed": "mixed varlen: 16 q / 4 kv heads, head 192 (b=64, n=3), block 16, 8 causal prefills q=kv ~ U[512,2048] + 120 decodes kv ~ U[1024,16384], shuffled order",
    "long": "long-context decode: Llama-3-8B shape, 32 q / 8 kv heads, head 128, block 16, batch 256 x kv 32768",
}


# ---------------------------------------------------------------------------
# distributed plumbing (host side only)
# ---------------------------------------------------------------------------
def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("LOCAL_RANK", "0"))


def dist_setup(use_cuda: bool):
    import torch
    import torch.distributed as dist
    rank, world, local = dist_env()
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if use_cuda else "gloo"
        if use_cuda:
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def replica_seed(base_seed: int, rank: int) -> int:
    """Each rank draws its own replica of the workload (weak scaling)."""
    return base_seed + 7919 * rank


def barrier(device):
    import torch
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        if device is not None and str(device).startswith("cuda"):
            dist.barrier(device_ids=[torch.cuda.current_device()])
        else:
            dist.barrier()


def max_over_ranks(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(units_per_rank: float, world: int, seconds_max: float) -> float:
    """Whole-job throughput: every rank's units over the slowest rank's time."""
    return units_per_rank * world / seconds_max


# ---------------------------------------------------------------------------
# measurement helpers
# ---------------------------------------------------------------------------
def load_peaks():
    """(HBM GB/s, bf16 dense TFLOP/s sustained, source) from MEASURED_PEAKS.json."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops_sustained", FALLBACK_TC_TFLOPS)), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_TC_TFLOPS, "fallback"


def decode_columns(w) -> int:
    """Query columns per key block of the decode kernel, as the library picks
    them: q_len * G of the longest query when every sequence fits in 8 columns,
    else G (longer queries go to prefill); two blocks share the 8 MMA columns
    when that count is at most 4."""
    mq = max(1, w.max_query_len) * w.group
    cols = mq if mq <= 8 else w.group
    return 4 if cols <= 4 else 8


NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, nominal (context only; `peak` is the measured copy)


def source_sha(paths) -> str:
    """First 16 hex digits of the SHA-256 of the files' bytes, in order."""
    h = hashlib.sha256()
    for path in paths:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_traffic_{workload}.txt")
    if not os.path.exists(path):
        return None
    kv = {}
    with open(path) as f:
        for line in f:
            if "=" in line and not line.startswith("#"):
                k, v = line.split("=", 1)
                kv[k.strip()] = v.strip()
    names = kv.get("source", "").split()
    srcs = [os.path.join(ROOT, "int4_token_head_gb300", "csrc", n) for n in names]
    if not srcs or not all(os.path.exists(p) for p in srcs) or kv.get("source_sha") != source_sha(srcs):
        return None
    try:
        return float(kv["bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_id: str, period_ms: int = 50):
        self.cmd = ["nvidia-smi", f"--id={gpu_id}", "--query-gpu=" + ",".join(self.FIELDS),
                    "--format=csv,noheader,nounits", "-lms", str(period_ms)]
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def gpu_id_for_smi(dev_index: int) -> str:
    import torch
    try:
        u = torch.cuda.get_device_properties(dev_index).uuid
        s = str(u)
        return s if s.startswith("GPU-") else "GPU-" + s
    except Exception:
        return str(dev_index)


def bulk_write_bench(w, dev, n_chunks: int, chunk_tokens: int = 65536, fmt: str = "int4"):
    """RHT + quantise write throughput: n_chunks pre-drawn 65,536-token chunks of
    this workload's shape (bf16 K and V, random slots of a scratch cache; the
    inputs, 2 x 65,536 x Hkv x d x 2 bytes per chunk, exceed L2) written back
    to back; one warm-up pass, then device time of a second pass by CUDA
    events.  Algorithmic bytes: bf16 K,V in + codes and scales out + slots.
    fmt "int8": the int8_per_token_head write (no rotation, d code bytes)."""
    import torch
    from int4_token_head_gb300 import _lib
    hkv, d, bs = w.num_kv_heads, w.head_size, w.block_size
    nb = chunk_tokens // bs
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed * 7 + 3)
    ks = [torch.randn((chunk_tokens, hkv, d), generator=g, device=dev).to(torch.bfloat16) for _ in range(n_chunks)]
    vs = [torch.randn((chunk_tokens, hkv, d), generator=g, device=dev).to(torch.bfloat16) for _ in range(n_chunks)]
    slots = [torch.randperm(nb * bs, generator=g, device=dev) for _ in range(n_chunks)]
    cb = d if fmt == "int8" else d // 2
    kc = torch.empty((nb, bs, hkv, cb), dtype=torch.int8 if fmt == "int8" else torch.uint8, device=dev)
    vc = torch.empty_like(kc)
    ksc = torch.empty((nb, bs, hkv), dtype=torch.float32, device=dev)
    vsc = torch.empty_like(ksc)
    signs = w.signs.to(dev)

    def one(i):
        if fmt == "int8":
            _lib.write_int8(ks[i], vs[i], slots[i], kc, vc, ksc, vsc)
        else:
            _lib.write(ks[i], vs[i], slots[i], kc, vc, ksc, vsc, signs)
    for i in range(n_chunks):
        one(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(n_chunks):
        one(i)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n_chunks
    nbytes = chunk_tokens * (2 * hkv * d * 2 + 2 * hkv * (cb + 4) + 8)
    del ks, vs, slots, kc, vc, ksc, vsc
    return {"gbs": round(nbytes / (ms / 1e3) / 1e9, 1), "ms_per_chunk": round(ms, 4), "chunks": n_chunks,
            "tokens_per_chunk": chunk_tokens, "bytes_per_chunk": nbytes}


def rht_bench(w, dev, n_chunks: int, chunk_tokens: int = 65536):
    """Standalone rotation (kv_int4_rht) throughput: n_chunks pre-drawn
    65,536-token x Hkv-head bf16 K chunks rotated to bf16, back to back;
    one warm-up pass, then device time of a second pass by CUDA events.
    Algorithmic bytes: bf16 in + bf16 out."""
    import torch
    from int4_token_head_gb300 import _lib
    hkv, d = w.num_kv_heads, w.head_size
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed * 7 + 5)
    xs = [torch.randn((chunk_tokens * hkv, d), generator=g, device=dev).to(torch.bfloat16) for _ in range(n_chunks)]
    ys = [torch.empty_like(x) for x in xs]
    signs = w.signs.to(dev)
    for x, y in zip(xs, ys):
        _lib.rht(x, signs, out=y)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for x, y in zip(xs, ys):
        _lib.rht(x, signs, out=y)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n_chunks
    nbytes = chunk_tokens * hkv * d * 2 * 2
    del xs, ys
    return {"gbs": round(nbytes / (ms / 1e3) / 1e9, 1), "ms_per_chunk": round(ms, 4), "chunks": n_chunks,
            "rows_per_chunk": chunk_tokens * hkv, "bytes_per_chunk": nbytes}


def window_bench(pk, q, out, window: int, iters: int):
    """Sliding-window attention over the resident cache: device time of
    `iters` back-to-back kv_int4_attention calls with the window, and the
    algorithmic bytes the window keeps (the last min(L, W + q_len - 1) keys
    of each sequence, their scales, q and the block table entries)."""
    import torch
    w = pk.w
    saved = w.sliding_window
    w.sliding_window = window
    try:
        pk.attend(q, out)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(iters):
            pk.attend(q, out)
        e1.record()
        torch.cuda.synchronize()
        if pk.status.item() != 0:
            raise RuntimeError(f"device status {pk.status.item()} in the windowed attention")
    finally:
        w.sliding_window = saved
    ms = e0.elapsed_time(e1) / iters
    d, hkv, hq = w.head_size, w.num_kv_heads, w.num_q_heads
    nbytes = 0
    for ql, L in w.seqs:
        keys = min(L, window + ql - 1)
        nbytes += keys * hkv * 2 * (d // 2 + 4) + 4 * ((keys + 15) // 16) + ql * hq * d * 2
    return {"window": window, "ms": round(ms, 5), "gbs": round(nbytes / (ms / 1e3) / 1e9, 1),
            "algorithmic_bytes": nbytes}


def prefill_kernel_name(d: int) -> str:
    """Head sizes up to 192 take the warp-specialised tcgen05 prefill, 256 the mma.sync one."""
    return "prefill_ws_kernel" if d <= 192 else "prefill_kernel"


def decode_kernel_name(d: int, int8: bool = False) -> str:
    """INT4 head size 128 has its own decode entry point (128 registers a thread)."""
    return "decode_kernel_i4d128" if d == 128 and not int8 else "decode_kernel"


def int8_decode_bench(w, dev, iters: int):
    """The int8_per_token_head mode on this workload: a second cache (int8
    codes, no rotation) populated through kv_int8_write, then `iters`
    attention calls; decode kernel time from the library's timer.
    Algorithmic bytes as for INT4 with d code bytes per head vector."""
    import torch
    from int4_token_head_gb300 import _lib
    from int4_token_head_gb300.paged import PagedKV
    pk = PagedKV(w, device=str(dev), fmt="int8")
    pk.populate_history(chunk_tokens=65536)
    q, k_new, v_new, slots = pk.step_inputs()
    out = torch.empty((w.num_q_tokens, w.num_q_heads, w.head_size), dtype=torch.bfloat16, device=dev)
    pk.step(q, k_new, v_new, slots, out)
    for _ in range(3):
        pk.attend(q, out)
    torch.cuda.synchronize()
    _lib.timing_collect()
    _lib.timing_enable(True)
    for _ in range(iters):
        pk.attend(q, out)
    torch.cuda.synchronize()
    kern = _lib.timing_collect()
    _lib.timing_enable(False)
    if pk.status.item() != 0:
        raise RuntimeError(f"device status {pk.status.item()} in the int8 attention")
    d, hkv, hq = w.head_size, w.num_kv_heads, w.num_q_heads
    dom = "decode" if kern["decode"][0] >= kern["prefill"][0] else "prefill"
    ms = kern[dom][0] / max(1, kern[dom][1])
    nbytes = sum(kv * hkv * 2 * (d + 4) + 4 * ((kv + 15) // 16) + ql * hq * d * 2 for ql, kv in w.seqs)
    step_ms = sum(kern[k][0] for k in ("prep", "prefill", "decode", "reduce")) / iters
    del pk
    torch.cuda.empty_cache()
    return {"kernel": prefill_kernel_name(w.head_size) if dom == "prefill" else decode_kernel_name(w.head_size, True),
            "ms": round(ms, 5),
            "attention_ms": round(step_ms, 5),
            "gbs": round(nbytes / (ms / 1e3) / 1e9, 1) if dom == "decode" else None,
            "cache_bytes_read": nbytes}


def inslot_bench(w, dev, pk, q, out, n_chunks: int, iters: int, chunk_tokens: int = 65536):
    """The in-slot scale layout (uint8 [blocks][2][16][Hkv][P], the scale
    inside every P-byte slot) for the INT4 format: bulk writes into an in-slot
    scratch cache, and decode over the resident cache repacked into that
    layout on the device (untimed).  Algorithmic bytes are the method's (the
    same as for the separate layout); the padding to P bytes is layout
    overhead, reported as slot_bytes."""
    import torch
    from int4_token_head_gb300 import _lib
    hkv, d, bs = w.num_kv_heads, w.head_size, w.block_size
    cb, P = d // 2, _lib.inslot_slot_bytes(d)
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed * 7 + 9)
    nb = chunk_tokens // bs
    ks = [torch.randn((chunk_tokens, hkv, d), generator=g, device=dev).to(torch.bfloat16) for _ in range(n_chunks)]
    vs = [torch.randn((chunk_tokens, hkv, d), generator=g, device=dev).to(torch.bfloat16) for _ in range(n_chunks)]
    slots = [torch.randperm(nb * bs, generator=g, device=dev) for _ in range(n_chunks)]
    scratch = torch.zeros((nb, 2, bs, hkv, P), dtype=torch.uint8, device=dev)
    signs = w.signs.to(dev)
    for i in range(n_chunks):
        _lib.write_inslot(ks[i], vs[i], slots[i], scratch, signs=signs)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(n_chunks):
        _lib.write_inslot(ks[i], vs[i], slots[i], scratch, signs=signs)
    e1.record()
    torch.cuda.synchronize()
    wms = e0.elapsed_time(e1) / n_chunks
    wbytes = chunk_tokens * (2 * hkv * d * 2 + 2 * hkv * (cb + 4) + 8)
    del ks, vs, slots, scratch
    # decode over the repacked resident cache
    NB = pk.k_cache.shape[0]
    ins = torch.zeros((NB, 2, bs, hkv, P), dtype=torch.uint8, device=dev)
    ins[:, 0, :, :, :cb] = pk.k_cache
    ins[:, 1, :, :, :cb] = pk.v_cache
    ins[:, 0, :, :, cb:cb + 4] = pk.k_scale.view(torch.uint8).view(NB, bs, hkv, 4)
    ins[:, 1, :, :, cb:cb + 4] = pk.v_scale.view(torch.uint8).view(NB, bs, hkv, 4)

    def attend():
        _lib.attention_inslot(q, ins, pk.block_table, pk.seq_lens, pk.query_start_loc, w.max_query_len,
                              w.max_seq_len, pk.softmax_scale, w.causal, out, pk.workspace, signs=pk.signs,
                              dev_status=pk.status, sliding_window=w.sliding_window)
    for _ in range(3):
        attend()
    torch.cuda.synchronize()
    _lib.timing_collect()
    _lib.timing_enable(True)
    for _ in range(iters):
        attend()
    torch.cuda.synchronize()
    kern = _lib.timing_collect()
    _lib.timing_enable(False)
    if pk.status.item() != 0:
        raise RuntimeError(f"device status {pk.status.item()} in the in-slot attention")
    del ins
    torch.cuda.empty_cache()
    res = {"slot_bytes": P, "write": {"gbs": round(wbytes / (wms / 1e3) / 1e9, 1), "ms_per_chunk": round(wms, 4)}}
    if kern["decode"][0] >= kern["prefill"][0] and kern["decode"][1]:
        dms = kern["decode"][0] / kern["decode"][1]
        dbytes = sum(kv * hkv * 2 * (cb + 4) + 4 * ((kv + 15) // 16) + ql * w.num_q_heads * d * 2
                     for ql, kv in w.seqs)
        res["decode"] = {"ms": round(dms, 5), "gbs": round(dbytes / (dms / 1e3) / 1e9, 1)}
    return res


# ---------------------------------------------------------------------------
# the oracle on host cores (CPU baseline and the reference arm)
# ---------------------------------------------------------------------------
def _unit_picks(w, n_units: int):
    """n_units (sequence, kv head) units spread evenly over the batch."""
    order = [(s, h) for s in range(w.num_seqs) for h in range(w.num_kv_heads)]
    stride = max(1, len(order) // max(1, n_units))
    return order[::stride][:n_units]


def _oracle_proc(rank, name, batch, picks, seconds, fixed_steps, warmup, chunk_tokens, gate, results):
    """One host process of the CPU oracle runner (spawned; never touches a GPU).

    Set-up (untimed): the oracle writes the history of its (sequence, kv
    head) units into caches of their own.  Timed, after every process has
    reached the gate: unit steps, each the oracle's write of the unit's new
    token plus its attention for the unit's q heads (fixed_steps of them, or
    as many as fit in `seconds`), then, after the gate again, the oracle's
    write of this process's share of one chunk of new tokens."""
    import numpy as np
    import torch
    torch.set_num_threads(1)
    from int4_token_head_gb300 import synthetic
    from oracle import kvint4_oracle as O
    try:
        overrides = {"batch": batch} if batch else {}
        w = synthetic.make_workload(name, **overrides)
        signs = w.signs.numpy()
        bs, d, hkv = w.block_size, w.head_size, w.num_kv_heads
        q_all = w.queries("cpu").float().numpy()
        qsl = w.query_start_loc.numpy()
        units = []
        drawn = {}
        for s, h in picks:
            ql, L = w.seqs[s]
            if s not in drawn:
                drawn.clear()
                k, v = w.seq_kv(s, "cpu")
                drawn[s] = (k.float().numpy(), v.float().numpy())
            k, v = drawn[s]
            k, v = k[:, h:h + 1], v[:, h:h + 1]
            nblk = (L + bs - 1) // bs
            kc = np.full((nblk, bs, 1, d // 2), 0xA5, np.uint8)
            vc = kc.copy()
            ks = np.full((nblk, bs, 1), np.nan, np.float32)
            vs = ks.copy()
            O.write_cache(k[:L - ql], v[:L - ql], np.arange(L - ql), kc, vc, ks, vs, bs, signs)
            q = q_all[qsl[s]:qsl[s + 1], h * w.group:(h + 1) * w.group]
            units.append((k[L - ql:].copy(), v[L - ql:].copy(), np.arange(L - ql, L), (kc, vc, ks, vs), q, L, ql,
                          nblk))
        drawn.clear()
        scale = 1.0 / math.sqrt(d)

        def step(i):
            k_new, v_new, slots, (kc, vc, ks, vs), q, L, ql, nblk = units[i % len(units)]
            O.write_cache(k_new, v_new, slots, kc, vc, ks, vs, bs, signs)
            O.attention_seq(q, kc, vc, ks, vs, np.arange(nblk)[None], [L], [0, ql], 0, 1, bs, scale, w.causal, signs)

        for i in range(warmup):
            step(i)
        # this process's share of one write chunk: bf16-representable N(0, 1) K/V, random slots
        rng = np.random.default_rng(1000 + rank)
        ck = rng.standard_normal((chunk_tokens, hkv, d)).astype(np.float32)
        cv = rng.standard_normal((chunk_tokens, hkv, d)).astype(np.float32)
        ck = (ck.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)
        cv = (cv.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)
        nb = max(1, (chunk_tokens + bs - 1) // bs)
        cache = [np.zeros((nb, bs, hkv, d // 2), np.uint8), np.zeros((nb, bs, hkv, d // 2), np.uint8),
                 np.zeros((nb, bs, hkv), np.float32), np.zeros((nb, bs, hkv), np.float32)]
        cslots = rng.permutation(nb * bs)[:chunk_tokens]
        gate.wait()
        t0 = time.perf_counter()
        n = 0
        while True:
            step(n)
            n += 1
            if fixed_steps is not None:
                if n >= fixed_steps:
                    break
            elif time.perf_counter() - t0 >= seconds:
                break
        t1 = time.perf_counter()
        gate.wait()
        t2 = time.perf_counter()
        if chunk_tokens:
            O.write_cache(ck, cv, cslots, *cache, bs, signs)
        t3 = time.perf_counter()
        results.put((rank, n, t0, t1, t2, t3, None))
    except Exception as e:  # reported by the parent
        try:
            gate.abort()
        except Exception:
            pass
        results.put((rank, 0, 0.0, 0.0, 0.0, 0.0, repr(e)))


def run_oracle_on_host(name, batch, processes, units_per_process, seconds=0.0, fixed_steps=None, warmup=1,
                       chunk_tokens=65536):
    """Time the fp64 oracle on `processes` host processes at once (one BLAS
    thread each; spawned, so safe after CUDA is initialised).  Returns the
    unit steps and their wall time (first start to last end), their
    throughput in decode tokens/s (a (sequence, kv head) unit is 1/Hkv of a
    decode token), and the write of one chunk of chunk_tokens tokens split
    evenly over the processes, with its wall time and GB/s."""
    import multiprocessing as mp
    from int4_token_head_gb300 import synthetic
    overrides = {"batch": batch} if batch else {}
    w = synthetic.make_workload(name, **overrides)
    picks = _unit_picks(w, processes * units_per_process)
    processes = max(1, min(processes, len(picks)))
    per = [picks[r::processes] for r in range(processes)]
    share = [chunk_tokens // processes + (1 if r < chunk_tokens % processes else 0) for r in range(processes)]
    ctx = mp.get_context("spawn")
    gate = ctx.Barrier(processes)
    results = ctx.Queue()
    keys = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
    saved = {k: os.environ.get(k) for k in keys}
    os.environ.update({k: "1" for k in keys})
    try:
        procs = [ctx.Process(target=_oracle_proc, args=(r, name, batch, per[r], seconds, fixed_steps, warmup,
                                                        share[r], gate, results), daemon=True)
                 for r in range(processes)]
        for p in procs:
            p.start()
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    out = [results.get(timeout=1800) for _ in range(processes)]
    for p in procs:
        p.join(60)
    errs = [o[6] for o in out if o[6]]
    if errs:
        raise RuntimeError(f"oracle process failed: {errs[0]}")
    steps = sum(o[1] for o in out)
    wall = max(o[3] for o in out) - min(o[2] for o in out)
    wwall = max(o[5] for o in out) - min(o[4] for o in out)
    d, hkv = w.head_size, w.num_kv_heads
    wbytes = chunk_tokens * (2 * hkv * d * 2 + 2 * hkv * (d // 2 + 4) + 8)
    return {"w": w, "processes": processes, "units": len(picks), "unit_steps": steps, "wall_s": wall,
            "steps_per_process": min(o[1] for o in out),
            "tokens_per_s": steps / hkv / wall, "total_units": w.num_seqs * hkv,
            "write_chunk": {"tokens": chunk_tokens, "s": round(wwall, 3),
                            "gbs": round(wbytes / wwall / 1e9, 4) if wwall > 0 else None}}


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def oracle_sample_text(r) -> str:
    w = r["w"]
    step_s = r["total_units"] / (r["unit_steps"] / r["wall_s"])
    return (f"{r['processes']} processes at once (one per host core, 1 BLAS thread each) on {r['units']} of the "
            f"{r['total_units']} (sequence, kv head) units of this batch; a unit step is the oracle's write of the "
            f"unit's new token + attention for its {w.group} q heads over up to {w.max_seq_len} keys (1 unit = "
            f"1/{w.num_kv_heads} decode token); {r['unit_steps']} unit steps in {r['wall_s']:.1f} s, so one whole "
            f"step ({r['total_units']} units) would take {step_s:.1f} s; the write of one "
            f"{r['write_chunk']['tokens']}-token chunk took {r['write_chunk']['s']} s = "
            f"{r['write_chunk']['gbs']} GB/s")


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def run_ours(args):
    import torch
    from int4_token_head_gb300 import _lib, synthetic
    from int4_token_head_gb300.paged import PagedKV

    rank, world, local = dist_setup(use_cuda=True)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    _lib.load()
    overrides = {}
    if args.batch:
        overrides["batch"] = args.batch
    w = synthetic.make_workload(args.workload, **overrides)
    w = synthetic.make_workload(args.workload, seed=replica_seed(w.seed, rank), **overrides)
    pk = PagedKV(w, device=str(dev))

    pk.populate_history(chunk_tokens=65536)
    torch.cuda.synchronize()
    write_info = bulk_write_bench(w, dev, args.write_chunks)
    rht_info = rht_bench(w, dev, max(1, args.write_chunks))
    q, k_new, v_new, slots = pk.step_inputs()
    out = torch.empty((w.num_q_tokens, w.num_q_heads, w.head_size), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()

    for _ in range(args.warmup):
        pk.step(q, k_new, v_new, slots, out)
    torch.cuda.synchronize()
    if pk.status.item() != 0:
        raise RuntimeError(f"device status {pk.status.item()} during warm-up")

    # ---- device-timed region: inputs resident in HBM ----
    sampler = ClockSampler(gpu_id_for_smi(local))
    barrier(dev)
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.2)
    _lib.timing_enable(True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        pk.step(q, k_new, v_new, slots, out)
    e1.record(stream)
    torch.cuda.synchronize()
    _lib.timing_enable(False)
    kern = _lib.timing_collect()
    clocks = sampler.stop()
    barrier(dev)
    ms_total = max_over_ranks(e0.elapsed_time(e1), dev)
    ms_step = ms_total / args.steps
    value = aggregate_throughput(w.num_q_tokens * args.steps, world, ms_total / 1e3)

    # ---- end to end through the C ABI with host buffers ----
    # Every step copies its inputs (queries, new K/V, slots, sequence
    # metadata) in from pinned host memory and its output back out, inside
    # the timed region.  The copies run on a second stream into two sets of
    # device buffers, so that the next step's inputs and the last step's
    # output move while a step computes, as in a serving loop; events order
    # each buffer's reuse.
    # The inputs are packed into one pinned host buffer (one copy in per
    # step), each field at a 256-byte aligned offset.
    fields = (q, k_new, v_new, slots, pk.seq_lens, pk.query_start_loc)
    nbytes = [t.numel() * t.element_size() for t in fields]
    offs, off = [], 0
    for n in nbytes:
        off = (off + 255) // 256 * 256
        offs.append(off)
        off += n
    h_in = torch.empty(off, dtype=torch.uint8).pin_memory()
    for t, o, n in zip(fields, offs, nbytes):
        h_in[o:o + n].copy_(t.detach().contiguous().cpu().view(-1).view(torch.uint8))
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(nbytes)
    d2h = h_out.numel() * h_out.element_size()
    copy_stream = torch.cuda.Stream(device=dev)
    d_in = [torch.empty(off, dtype=torch.uint8, device=dev) for _ in range(2)]
    views = [[d[o:o + n].view(t.dtype).view(t.shape) for t, o, n in zip(fields, offs, nbytes)] + [torch.empty_like(out)]
             for d in d_in]
    in_ready, done, out_free = ([torch.cuda.Event(), torch.cuda.Event()] for _ in range(3))

    def copy_in(i):
        b = i % 2
        if i >= 2:
            copy_stream.wait_event(done[b])  # step i - 2 is done with this set
        with torch.cuda.stream(copy_stream):
            d_in[b].copy_(h_in, non_blocking=True)
        in_ready[b].record(copy_stream)

    def compute(i):
        b = i % 2
        d_q, d_k, d_v, d_s, d_sl, d_qsl, d_out = views[b]
        stream.wait_event(in_ready[b])
        if i >= 2:
            stream.wait_event(out_free[b])  # step i - 2's output has been copied out
        _lib.write(d_k, d_v, d_s, pk.k_cache, pk.v_cache, pk.k_scale, pk.v_scale, pk.signs,
                   dev_status=pk.status, stream=stream)
        _lib.attention(d_q, pk.k_cache, pk.v_cache, pk.k_scale, pk.v_scale, pk.block_table, d_sl, d_qsl,
                       w.max_query_len, w.max_seq_len, pk.softmax_scale, w.causal, pk.signs, d_out, pk.workspace,
                       dev_status=pk.status, stream=stream, sliding_window=w.sliding_window)
        done[b].record(stream)

    def copy_out(i):
        b = i % 2
        copy_stream.wait_event(done[b])
        with torch.cuda.stream(copy_stream):
            h_out.copy_(views[b][6], non_blocking=True)
        out_free[b].record(copy_stream)

    def e2e_run(n):
        copy_in(0)
        for i in range(n):
            if i + 1 < n:
                copy_in(i + 1)
            compute(i)
            copy_out(i)
        stream.wait_stream(copy_stream)  # the last output is on the host

    copy_stream.wait_stream(stream)
    e2e_run(max(1, args.warmup))
    torch.cuda.synchronize()
    barrier(dev)
    torch.cuda.synchronize()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    copy_stream.wait_stream(stream)  # the first copy starts after f0
    e2e_run(args.steps)
    f1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(f0.elapsed_time(f1), dev)
    e2e_value = aggregate_throughput(w.num_q_tokens * args.steps, world, e2e_ms / 1e3)
    if pk.status.item() != 0:
        raise RuntimeError(f"device status {pk.status.item()} during the timed region")
    # the same inputs and cache give the same bits: the end-to-end loop did the whole step
    if not torch.equal(h_out, out.cpu()):
        raise RuntimeError("the end-to-end loop's output differs from the device-timed loop's")
    window_info = window_bench(pk, q, out, 4096, max(10, min(200, args.steps)))
    inslot_info = inslot_bench(w, dev, pk, q, out, max(1, args.write_chunks), max(10, min(200, args.steps)))
    int8_info = {"write": bulk_write_bench(w, dev, max(1, args.write_chunks), fmt="int8")}
    int8_info.update(int8_decode_bench(w, dev, max(10, min(200, args.steps))))

    # ---- roofline of the dominant kernel ----
    peak, tc_peak, peak_kind = load_peaks()
    dom = max(("decode", "prefill"), key=lambda k: kern[k][0])
    dom_ms, dom_n, _ = kern[dom]
    d, hkv, hq = w.head_size, w.num_kv_heads, w.num_q_heads
    dcols = decode_columns(w)
    is_dec = lambda ql: w.group <= dcols and ql * w.group <= dcols
    launch_s = dom_ms / dom_n / 1e3 if dom_n else None
    if dom == "decode":
        seqs = [(ql, kv) for ql, kv in w.seqs if is_dec(ql)]
        algo = sum(kv * hkv * 2 * (d // 2 + 4) + 4 * ((kv + 15) // 16) + ql * hq * d * 2 for ql, kv in seqs)
        achieved = algo / launch_s / 1e9 if launch_s else None
        roofline = {"bound": "hbm", "achieved": round(achieved, 1) if achieved else None, "peak": peak,
                    "unit": "GB/s", "frac": round(achieved / peak, 4) if achieved else None,
                    "traffic": recorded_traffic(dom, args.workload), "kernel": decode_kernel_name(d),
                    "peak_source": f"{peak_kind} (HBM copy)", "algorithmic_bytes_per_launch": algo,
                    "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4) if achieved else None,
                    "nominal_peak": NOMINAL_HBM_GBS}
    else:
        # a dense contraction: QK^T and PV over the visible (query, key) pairs
        seqs = [(ql, kv) for ql, kv in w.seqs if not is_dec(ql)]
        pairs = sum((ql * (kv - ql) + ql * (ql + 1) // 2) if w.causal else ql * kv for ql, kv in seqs)
        flops = 4 * d * hq * pairs
        achieved = flops / launch_s / 1e12 if launch_s else None
        roofline = {"bound": "tensor", "achieved": round(achieved, 2) if achieved else None, "peak": tc_peak,
                    "unit": "TFLOP/s", "frac": round(achieved / tc_peak, 4) if achieved else None,
                    "traffic": recorded_traffic(dom, args.workload), "kernel": prefill_kernel_name(d),
                    "peak_source": f"{peak_kind} bf16 dense, sustained (cuBLAS); f16 has the same nominal rate",
                    "algorithmic_flops_per_launch": flops}
    roofline["avg_launch_ms"] = round(dom_ms / dom_n, 5) if dom_n else None

    # whole-attention and write throughput
    attn_bytes = pk.kv_bytes_read()
    attn_ms = sum(kern[k][0] for k in ("prep", "prefill", "decode", "reduce")) / args.steps
    write_info["frac"] = round(write_info["gbs"] / peak, 4)
    write_info["step_write_us"] = round(kern["write"][0] / max(1, kern["write"][1]) * 1e3, 2)
    rht_info["frac"] = round(rht_info["gbs"] / peak, 4)
    window_info["frac"] = round(window_info["gbs"] / peak, 4)
    int8_info["write"]["frac"] = round(int8_info["write"]["gbs"] / peak, 4)
    inslot_info["write"]["frac"] = round(inslot_info["write"]["gbs"] / peak, 4)
    if "decode" in inslot_info:
        inslot_info["decode"]["frac"] = round(inslot_info["decode"]["gbs"] / peak, 4)
    if int8_info["gbs"]:
        int8_info["frac"] = round(int8_info["gbs"] / peak, 4)

    result = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int4 codes, f16 mma / f32 accumulate, f32 rotation",
        "data": "synthetic (seeded N(0,1) bf16 K/V/Q; no dataset or weights)",
        "config": bench_config(args, w, world),
        "roofline": roofline,
        "kv_read_gbs": round(attn_bytes / (attn_ms / 1e3) / 1e9, 1) if attn_ms else None,
        "write": write_info,
        "rht": rht_info,
        "sliding_window": window_info,
        "int8_per_token_head": int8_info,
        "inslot_scales": inslot_info,
        "kernels_ms_per_step": {k: round(v[0] / args.steps, 5) for k, v in kern.items()},
        "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": int(sum(v[1] for v in kern.values())),
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        r = run_oracle_on_host(args.workload, args.batch, host_cores(), units_per_process=2,
                               seconds=args.cpu_seconds, warmup=1)
        result["cpu_baseline"] = {"value": round(r["tokens_per_s"], 3), "unit": UNIT, "cores": r["processes"],
                                  "kind": "oracle", "sample": oracle_sample_text(r),
                                  "write_chunk_gbs": r["write_chunk"]["gbs"]}
    if rank == 0:
        print(json.dumps(result), flush=True)


# ---------------------------------------------------------------------------
# reference arm: the oracle on host cores
# ---------------------------------------------------------------------------
def run_reference(args):
    """The reference arm: the fp64 oracle on the host cores (rank 0 only),
    each step one unit step (write of a new token + attention of one
    (sequence, kv head) unit) in every host process at once."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    r = run_oracle_on_host(args.workload, args.batch, host_cores(), units_per_process=1, fixed_steps=args.steps,
                           warmup=args.warmup)
    w = r["w"]
    v = r["tokens_per_s"]
    result = {
        "impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(r["wall_s"] / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) bf16 K/V/Q; no dataset or weights)",
        "config": bench_config(args, w, world),
        "cpu_baseline": {"value": round(v, 4), "unit": UNIT, "cores": r["processes"], "kind": "oracle",
                         "sample": oracle_sample_text(r), "write_chunk_gbs": r["write_chunk"]["gbs"]},
        "e2e": {"value": round(v, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(result), flush=True)


def bench_config(args, w, world):
    """The workload description both arms print (identical for the same arguments)."""
    cache_gb = w.num_blocks * w.block_size * w.num_kv_heads * (w.head_size + 8) / 1e9
    return {"workload": WORKLOAD_TEXT[args.workload], "name": args.workload,
            "global_batch": w.num_seqs * world, "seq_len": w.max_seq_len,
            "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
            "collectives": "none on the data path (replicas; a barrier and a max over ranks around the timing)",
            "l2": "inputs larger than L2 (cache %.2f GB), no flush" % cache_gb}


def launch_replicas(n: int, argv) -> int:
    """`--gpus N` without a surrounding launcher: run this script under
    torch.distributed.run with N ranks on this node (one replica per GPU)."""
    import socket
    if "--impl" not in argv or argv[argv.index("--impl") + 1] != "reference":
        import torch
        if torch.cuda.device_count() < n:
            print(f"bench.py --gpus {n} needs {n} visible GPUs; {torch.cuda.device_count()} found", file=sys.stderr)
            return 2
    sock = socket.socket()
    sock.bind(("127.0.0.1", 0))
    port = sock.getsockname()[1]
    sock.close()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr=127.0.0.1", f"--master-port={port}", os.path.abspath(__file__), *argv]
    return subprocess.call(cmd)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOAD_TEXT), default="long")
    ap.add_argument("--batch", type=int, default=0, help="override the batch size (reduced-size cases)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--write-chunks", type=int, default=16, help="65,536-token chunks in the bulk write measurement")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    argv = list(sys.argv[1:] if argv is None else argv)
    args = ap.parse_args(argv)
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(launch_replicas(args.gpus, argv))
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
