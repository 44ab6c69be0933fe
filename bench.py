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

prints one JSON line.  Under torchrun (N > 1) every rank runs its own
replica of the workload (weak scaling, no collective on the data path); the
timed region is bracketed by a barrier and synchronize on every rank and
the slowest rank's time is used.

--impl reference times the fp64 CPU oracle on the host cores (rank 0 only)
on a bounded sample of the same workload: each step is the oracle's write of
one new token plus its attention for one (sequence, kv head) unit of the
batch, i.e. 1/num_kv_heads of a decode token.
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
class OracleUnits:
    """A pool of (sequence, kv head) units of the workload, each with its own
    oracle-written cache; a step is the oracle's write of the unit's new
    token plus its attention for the unit's q heads."""

    def __init__(self, w, n_units: int, gen_device: str):
        import numpy as np
        from oracle import kvint4_oracle as O
        self.O, self.np = O, np
        self.w = w
        self.units = []
        q_all = w.queries(gen_device).float().cpu().numpy()
        qsl = w.query_start_loc.numpy()
        order = [(s, h) for s in range(w.num_seqs) for h in range(w.num_kv_heads)]
        stride = max(1, len(order) // max(1, n_units))
        picks = order[::stride][:n_units]
        for s, h in picks:
            ql, L = w.seqs[s]
            k, v = w.seq_kv(s, gen_device)
            k = k[:, h:h + 1].float().cpu().numpy()
            v = v[:, h:h + 1].float().cpu().numpy()
            nblk = (L + w.block_size - 1) // w.block_size
            kc = np.full((nblk, w.block_size, 1, w.head_size // 2), 0xA5, np.uint8)
            vc = kc.copy()
            ks = np.full((nblk, w.block_size, 1), np.nan, np.float32)
            vs = ks.copy()
            O.write_cache(k[:L - ql], v[:L - ql], np.arange(L - ql), kc, vc, ks, vs, w.block_size,
                          w.signs.numpy())
            q = q_all[qsl[s]:qsl[s + 1], h * w.group:(h + 1) * w.group]
            self.units.append(dict(k_new=k[L - ql:], v_new=v[L - ql:], slots=np.arange(L - ql, L),
                                   caches=(kc, vc, ks, vs), q=q, L=L, ql=ql, nblk=nblk))

    def step(self, i: int):
        u = self.units[i % len(self.units)]
        O, np, w = self.O, self.np, self.w
        kc, vc, ks, vs = u["caches"]
        O.write_cache(u["k_new"], u["v_new"], u["slots"], kc, vc, ks, vs, w.block_size, w.signs.numpy())
        return O.attention_seq(u["q"], kc, vc, ks, vs, np.arange(u["nblk"])[None], [u["L"]], [0, u["ql"]], 0, 1,
                               w.block_size, 1.0 / math.sqrt(w.head_size), w.causal, w.signs.numpy())


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def time_oracle(w, gen_device, max_seconds: float, min_steps: int = 3, fixed_steps=None, warmup: int = 1,
                n_units: int = 2):
    pool = OracleUnits(w, n_units, gen_device)
    for i in range(warmup):
        pool.step(i)
    t0 = time.perf_counter()
    n = 0
    while True:
        pool.step(n)
        n += 1
        el = time.perf_counter() - t0
        if fixed_steps is not None:
            if n >= fixed_steps:
                break
        elif n >= min_steps and el >= max_seconds:
            break
    el = time.perf_counter() - t0
    tokens = n / w.num_kv_heads
    return tokens / el, n, el, pool


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
    pin = lambda t: t.cpu().pin_memory()
    h_q, h_k, h_v, h_s = pin(q), pin(k_new), pin(v_new), pin(slots)
    h_sl, h_qsl = pin(pk.seq_lens), pin(pk.query_start_loc)
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    d_q, d_k, d_v, d_s = torch.empty_like(q), torch.empty_like(k_new), torch.empty_like(v_new), torch.empty_like(slots)
    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_k, h_v, h_s, h_sl, h_qsl))
    d2h = h_out.numel() * h_out.element_size()

    def e2e_step():
        d_q.copy_(h_q, non_blocking=True)
        d_k.copy_(h_k, non_blocking=True)
        d_v.copy_(h_v, non_blocking=True)
        d_s.copy_(h_s, non_blocking=True)
        pk.seq_lens.copy_(h_sl, non_blocking=True)
        pk.query_start_loc.copy_(h_qsl, non_blocking=True)
        pk.step(d_q, d_k, d_v, d_s, out)
        h_out.copy_(out, non_blocking=True)

    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    barrier(dev)
    torch.cuda.synchronize()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    f1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(f0.elapsed_time(f1), dev)
    e2e_value = aggregate_throughput(w.num_q_tokens * args.steps, world, e2e_ms / 1e3)
    if pk.status.item() != 0:
        raise RuntimeError(f"device status {pk.status.item()} during the timed region")
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
        "config": {"workload": WORKLOAD_TEXT[args.workload], "name": args.workload,
                   "global_batch": w.num_seqs * world, "seq_len": w.max_seq_len,
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                   "l2": "inputs larger than L2 (cache %.2f GB), no flush" % (
                       (pk.k_cache.numel() * 2 + pk.k_scale.numel() * 8) / 1e9)},
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
        v, n, el, _ = time_oracle(w, str(dev), max_seconds=args.cpu_seconds)
        result["cpu_baseline"] = {"value": round(v, 3), "unit": UNIT, "cores": host_cores(), "kind": "oracle",
                                  "sample": f"{n} (sequence, kv head) units of this batch, each the oracle's "
                                            f"write of one new token + attention for its {w.group} q heads "
                                            f"over {w.max_seq_len} keys; {el:.1f} s; 1 unit = 1/{w.num_kv_heads} token"}
    if rank == 0:
        print(json.dumps(result), flush=True)


# ---------------------------------------------------------------------------
# reference arm: the oracle on host cores
# ---------------------------------------------------------------------------
def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import torch
    from int4_token_head_gb300 import synthetic
    overrides = {"batch": args.batch} if args.batch else {}
    w = synthetic.make_workload(args.workload, **overrides)
    gen = "cuda" if torch.cuda.is_available() else "cpu"
    v, n, el, _ = time_oracle(w, gen, max_seconds=0, fixed_steps=args.steps, warmup=args.warmup, n_units=4)
    result = {
        "impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / n * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) bf16 K/V/Q; no dataset or weights)",
        "config": {"workload": WORKLOAD_TEXT[args.workload], "name": args.workload,
                   "global_batch": w.num_seqs, "seq_len": w.max_seq_len, "parallelism": "host cores"},
        "cpu_baseline": {"value": round(v, 4), "unit": UNIT, "cores": host_cores(), "kind": "oracle",
                         "sample": f"each step: the oracle's write of one new token + attention for one "
                                   f"(sequence, kv head) unit ({w.group} q heads over {w.max_seq_len} keys), "
                                   f"cycling over 4 units; 1 unit = 1/{w.num_kv_heads} token"},
        "e2e": {"value": round(v, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(result), flush=True)


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
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
