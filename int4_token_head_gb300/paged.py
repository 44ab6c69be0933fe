"""Device-side state of a paged INT4 (or int8_per_token_head) KV cache for
one synthetic workload.

Allocates the sentinel-filled caches and metadata on the GPU, populates each
sequence's history through the library's write path, and runs the step
(write the step's new K/V, then attention).  It only moves tensors and calls
the library; all arithmetic is in libkvint4.so.
"""

from __future__ import annotations

import math
from typing import List, Optional

import torch

from . import _lib
from .synthetic import Workload


class PagedKV:
    def __init__(self, w: Workload, device: str = "cuda", fmt: str = "int4"):
        if fmt not in ("int4", "int8"):
            raise ValueError(f"unknown cache format {fmt!r}")
        self.w = w
        self.device = device
        self.fmt = fmt
        caches = w.empty_cache(device) if fmt == "int4" else w.empty_cache_int8(device)
        self.k_cache, self.v_cache, self.k_scale, self.v_scale = caches
        self.signs = w.signs.to(device)
        self.block_table = w.block_table.to(device)
        self.seq_lens = w.seq_lens.to(device)
        self.query_start_loc = w.query_start_loc.to(device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.softmax_scale = 1.0 / math.sqrt(w.head_size)
        ws = _lib.attention_workspace_size(w.num_seqs, w.num_q_tokens, w.num_q_heads, w.num_kv_heads, w.head_size)
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=device)

    # -------------------------------------------------------------------
    def write(self, k, v, slots, stream=None, prerotated=False):
        if self.fmt == "int8":
            if prerotated:
                raise ValueError("the int8 cache stores unrotated vectors")
            _lib.write_int8(k, v, slots, self.k_cache, self.v_cache, self.k_scale, self.v_scale,
                            dev_status=self.status, stream=stream)
            return
        _lib.write(k, v, slots, self.k_cache, self.v_cache, self.k_scale, self.v_scale, self.signs,
                   dev_status=self.status, stream=stream, prerotated=prerotated)

    def populate_history(self, gen_device: Optional[str] = None, chunk_tokens: int = 65536,
                         timer: Optional[List[float]] = None):
        """Write every sequence's history (positions before its queries).

        K/V are drawn per sequence on ``gen_device`` (default: the cache's
        device) and written in chunks of about ``chunk_tokens`` tokens.  If
        ``timer`` is a list, the device time of each write call (ms) and its
        token count are appended to it as (ms, tokens).
        """
        w = self.w
        gen_device = gen_device or self.device
        pend_k, pend_v, pend_s, n = [], [], [], 0

        def flush():
            nonlocal pend_k, pend_v, pend_s, n
            if not n:
                return
            k = torch.cat(pend_k).to(self.device)
            v = torch.cat(pend_v).to(self.device)
            s = torch.cat(pend_s).to(self.device)
            if timer is not None:
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                self.write(k, v, s)
                e1.record()
                e1.synchronize()
                timer.append((e0.elapsed_time(e1), int(k.shape[0])))
            else:
                self.write(k, v, s)
            pend_k, pend_v, pend_s, n = [], [], [], 0

        for s, (q, kv) in enumerate(w.seqs):
            if kv - q <= 0:
                continue
            k, v = w.seq_kv(s, gen_device, positions=(0, kv - q))
            pend_k.append(k)
            pend_v.append(v)
            pend_s.append(w.slots(s, 0, kv - q))
            n += k.shape[0]
            if n >= chunk_tokens:
                flush()
        flush()

    def step_inputs(self, gen_device: Optional[str] = None):
        """(q, k_new, v_new, slot_mapping) of one step, on the cache's device."""
        gen_device = gen_device or self.device
        q = self.w.queries(gen_device).to(self.device)
        k, v = self.w.step_kv(gen_device)
        return q, k.to(self.device), v.to(self.device), self.w.step_slot_mapping().to(self.device)

    def attend(self, q, out, stream=None):
        w = self.w
        if self.fmt == "int8":
            _lib.attention_int8(q, self.k_cache, self.v_cache, self.k_scale, self.v_scale, self.block_table,
                                self.seq_lens, self.query_start_loc, w.max_query_len, w.max_seq_len,
                                self.softmax_scale, w.causal, out, self.workspace, dev_status=self.status,
                                stream=stream, sliding_window=w.sliding_window)
            return
        _lib.attention(q, self.k_cache, self.v_cache, self.k_scale, self.v_scale, self.block_table,
                       self.seq_lens, self.query_start_loc, w.max_query_len, w.max_seq_len,
                       self.softmax_scale, w.causal, self.signs, out, self.workspace,
                       dev_status=self.status, stream=stream, sliding_window=w.sliding_window)

    def step(self, q, k_new, v_new, slots, out, stream=None):
        self.write(k_new, v_new, slots, stream=stream)
        self.attend(q, out, stream=stream)

    # -------------------------------------------------------------------
    def kv_bytes_read(self) -> int:
        """Algorithmic bytes of one attention call: packed codes + scales of
        every key read, block-table entries, Q in and O out, metadata."""
        w = self.w
        d, hkv, hq = w.head_size, w.num_kv_heads, w.num_q_heads
        total = 0
        for q, kv in w.seqs:
            total += kv * hkv * 2 * (d // 2 + 4)
            total += 4 * ((kv + w.block_size - 1) // w.block_size)
            total += q * hq * d * 2 * 2
            total += 12
        return total

    def write_bytes(self, num_tokens: int) -> int:
        """Algorithmic bytes of writing num_tokens tokens: bf16 K,V in, codes and scales out, slot ids."""
        w = self.w
        d, hkv = w.head_size, w.num_kv_heads
        return num_tokens * (2 * hkv * d * 2 + 2 * hkv * (d // 2 + 4) + 8)
