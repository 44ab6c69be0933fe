"""Seeded synthetic workloads for the INT4 per-token-head KV cache.

This module only draws inputs: random signs for the diagonal D, sequence
lengths, block tables, slot mappings and bf16 K/V/Q values.  It contains none
of the method's arithmetic (no rotation, no quantisation, no attention), so
that both the CUDA path and the CPU oracle can be fed from it.

Draw order for the metadata generator (``torch.Generator('cpu')`` seeded with
``seed``): signs -> lengths -> sequence order -> block permutation -> outlier
channels.  Token values are drawn per sequence from a generator seeded with
``seed * 100003 + seq_index`` (K then V), and queries from one seeded with
``seed * 100003 + 99991``, on whichever device the caller asks for.

The five workloads are the ones the method's pages discuss: a tiny causal
case shaped like the pages' INT4 attention test (block 16, head 128, two
sequences of (q, kv) = (4, 128), (4, 97)); a Phi-3-mini decode batch with a
non-power-of-two head (96); a Llama-3.2-1B GQA decode batch; a mixed varlen
batch with head 192; and a long-context Llama-3-8B decode batch.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional, Tuple

import torch

SENTINEL_CODE_BYTE = 0xA5
# A quiet-NaN bit pattern; any unmasked read of an unwritten scale slot turns
# the attention output into NaN, which the tests catch.
SENTINEL_SCALE_BITS = 0x7FC00A5A

CONFIG_NAMES = ("tiny", "phi3", "gqa", "mixed", "long")


@dataclasses.dataclass
class Workload:
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_size: int
    block_size: int
    causal: bool
    seed: int
    # per sequence (q_len, kv_len), in batch order
    seqs: List[Tuple[int, int]]
    num_blocks: int
    signs: torch.Tensor          # int8 [head_size], entries +-1
    block_table: torch.Tensor    # int32 [num_seqs, max_blocks_per_seq], -1 padded
    outlier_channels: Optional[torch.Tensor]  # int64 [n] flat (kv_head*d + ch)
    outlier_scale: float
    sliding_window: int = 0      # 0: none; else a query at p sees no key at p - W or before

    @property
    def num_seqs(self) -> int:
        return len(self.seqs)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def seq_lens(self) -> torch.Tensor:
        return torch.tensor([kv for _, kv in self.seqs], dtype=torch.int32)

    @property
    def query_lens(self) -> torch.Tensor:
        return torch.tensor([q for q, _ in self.seqs], dtype=torch.int32)

    @property
    def query_start_loc(self) -> torch.Tensor:
        ql = self.query_lens.to(torch.int64)
        out = torch.zeros(self.num_seqs + 1, dtype=torch.int32)
        out[1:] = torch.cumsum(ql, 0).to(torch.int32)
        return out

    @property
    def num_q_tokens(self) -> int:
        return int(sum(q for q, _ in self.seqs))

    @property
    def max_query_len(self) -> int:
        return int(max(q for q, _ in self.seqs))

    @property
    def max_seq_len(self) -> int:
        return int(max(kv for _, kv in self.seqs))

    def slots(self, seq: int, start: int, stop: int) -> torch.Tensor:
        """Slot ids (int64) of token positions [start, stop) of sequence ``seq``."""
        pos = torch.arange(start, stop, dtype=torch.int64)
        blk = self.block_table[seq].to(torch.int64)[pos // self.block_size]
        return blk * self.block_size + pos % self.block_size

    def history_slot_mapping(self) -> torch.Tensor:
        """Slots of every position before each sequence's queries, seq-major."""
        parts = [self.slots(s, 0, kv - q) for s, (q, kv) in enumerate(self.seqs)]
        return torch.cat(parts) if parts else torch.zeros(0, dtype=torch.int64)

    def step_slot_mapping(self) -> torch.Tensor:
        """Slots of the step's new tokens (the query positions), in query order."""
        parts = [self.slots(s, kv - q, kv) for s, (q, kv) in enumerate(self.seqs)]
        return torch.cat(parts) if parts else torch.zeros(0, dtype=torch.int64)

    def empty_cache(self, device="cpu"):
        """Sentinel-filled caches: codes 0xA5, scales a NaN payload."""
        nb, bs, h, d = self.num_blocks, self.block_size, self.num_kv_heads, self.head_size
        kc = torch.full((nb, bs, h, d // 2), SENTINEL_CODE_BYTE, dtype=torch.uint8, device=device)
        vc = torch.full_like(kc, SENTINEL_CODE_BYTE)
        ks = torch.full((nb, bs, h), SENTINEL_SCALE_BITS, dtype=torch.int32, device=device).view(torch.float32)
        vs = ks.clone()
        return kc, vc, ks, vs

    def empty_cache_int8(self, device="cpu"):
        """Sentinel-filled int8_per_token_head caches: codes 0xA5, scales a NaN payload."""
        nb, bs, h, d = self.num_blocks, self.block_size, self.num_kv_heads, self.head_size
        kc = torch.full((nb, bs, h, d), SENTINEL_CODE_BYTE, dtype=torch.uint8, device=device).view(torch.int8)
        vc = kc.clone()
        ks = torch.full((nb, bs, h), SENTINEL_SCALE_BITS, dtype=torch.int32, device=device).view(torch.float32)
        return kc, vc, ks, ks.clone()

    # ---- token values -------------------------------------------------
    def seq_kv(self, seq: int, device="cpu", positions: Optional[Tuple[int, int]] = None):
        """bf16 K and V [kv_len, Hkv, d] of every position of sequence ``seq``.

        Values are N(0, 1) rounded to bf16; outlier channels (if any) are
        multiplied by ``outlier_scale`` before the bf16 rounding.  When
        ``positions`` is given only that slice is returned (the whole sequence
        is still drawn so that values do not depend on the slice).
        """
        _, kv = self.seqs[seq]
        g = torch.Generator(device=device)
        g.manual_seed(self.seed * 100003 + seq)
        shape = (kv, self.num_kv_heads, self.head_size)
        k = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        v = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        if self.outlier_channels is not None and self.outlier_channels.numel():
            mult = torch.ones(self.num_kv_heads * self.head_size, device=device)
            mult[self.outlier_channels.to(device)] = self.outlier_scale
            mult = mult.view(1, self.num_kv_heads, self.head_size)
            k = k * mult
            v = v * mult
        k = k.to(torch.bfloat16)
        v = v.to(torch.bfloat16)
        if positions is not None:
            k = k[positions[0]:positions[1]]
            v = v[positions[0]:positions[1]]
        return k, v

    def queries(self, device="cpu") -> torch.Tensor:
        """bf16 Q [num_q_tokens, Hq, d], N(0, 1)."""
        g = torch.Generator(device=device)
        g.manual_seed(self.seed * 100003 + 99991)
        q = torch.randn((self.num_q_tokens, self.num_q_heads, self.head_size),
                        generator=g, device=device, dtype=torch.float32)
        return q.to(torch.bfloat16)

    def step_kv(self, device="cpu"):
        """bf16 K, V of the step's new tokens [num_q_tokens, Hkv, d], in query order."""
        ks, vs = [], []
        for s, (q, kv) in enumerate(self.seqs):
            if q == 0:
                continue
            k, v = self.seq_kv(s, device, positions=(kv - q, kv))
            ks.append(k)
            vs.append(v)
        shape = (0, self.num_kv_heads, self.head_size)
        if not ks:
            z = torch.zeros(shape, dtype=torch.bfloat16, device=device)
            return z, z.clone()
        return torch.cat(ks), torch.cat(vs)

    def history_kv(self, device="cpu"):
        """bf16 K, V of every history position (before the queries), seq-major."""
        ks, vs = [], []
        for s, (q, kv) in enumerate(self.seqs):
            k, v = self.seq_kv(s, device, positions=(0, kv - q))
            ks.append(k)
            vs.append(v)
        return torch.cat(ks), torch.cat(vs)


def _blocks(n: int, bs: int) -> int:
    return (n + bs - 1) // bs


def make_workload(name: str, seed: Optional[int] = None, **overrides) -> Workload:
    """Build one of the named workloads with its seeded metadata.

    ``overrides`` may replace ``batch`` (number of sequences) or ``kv_len``
    for the fixed-length decode workloads, to build reduced-size variants.
    """
    if name not in CONFIG_NAMES:
        raise ValueError(f"unknown workload {name!r}; expected one of {CONFIG_NAMES}")
    idx = CONFIG_NAMES.index(name) + 1
    if seed is None:
        seed = 1000 + idx
    g = torch.Generator("cpu")
    g.manual_seed(seed)

    bs = 16
    outlier_scale = 1.0
    spare = 16
    if name == "tiny":
        hq, hkv, d = 4, 4, 128
        spare = 1
    elif name == "phi3":
        hq, hkv, d = 32, 32, 96
    elif name == "gqa":
        hq, hkv, d = 32, 8, 128
    elif name == "mixed":
        hq, hkv, d = 16, 4, 192
    else:  # long
        hq, hkv, d = 32, 8, 128
        spare = 0

    signs = (torch.randint(0, 2, (d,), generator=g, dtype=torch.int64) * 2 - 1).to(torch.int8)

    if name == "tiny":
        seqs = [(4, 128), (4, 97)]
    elif name == "phi3":
        batch = overrides.get("batch", 32)
        kv = overrides.get("kv_len", 1024)
        seqs = [(1, kv)] * batch
    elif name == "gqa":
        batch = overrides.get("batch", 64)
        lo, hi = overrides.get("kv_range", (512, 8192))
        lens = torch.randint(lo, hi + 1, (batch,), generator=g)
        seqs = [(1, int(x)) for x in lens]
    elif name == "mixed":
        n_pre = overrides.get("prefills", 8)
        n_dec = overrides.get("decodes", 120)
        plo, phi = overrides.get("prefill_range", (512, 2048))
        dlo, dhi = overrides.get("decode_range", (1024, 16384))
        pl = torch.randint(plo, phi + 1, (n_pre,), generator=g)
        dl = torch.randint(dlo, dhi + 1, (n_dec,), generator=g)
        seqs = [(int(x), int(x)) for x in pl] + [(1, int(x)) for x in dl]
        order = torch.randperm(len(seqs), generator=g)
        seqs = [seqs[int(i)] for i in order]
    else:
        batch = overrides.get("batch", 256)
        kv = overrides.get("kv_len", 32768)
        seqs = [(1, kv)] * batch

    nblk = [_blocks(kv, bs) for _, kv in seqs]
    num_blocks = sum(nblk) + spare
    perm = torch.randperm(num_blocks, generator=g).to(torch.int32)
    max_blocks = max(nblk)
    table = torch.full((len(seqs), max_blocks), -1, dtype=torch.int32)
    off = 0
    for s, n in enumerate(nblk):
        table[s, :n] = perm[off:off + n]
        off += n

    outliers = None
    if name == "phi3":
        n_pairs = hkv * d
        n_out = round(0.01 * n_pairs)
        outliers = torch.randperm(n_pairs, generator=g)[:n_out]
        outlier_scale = 8.0

    return Workload(name=name, num_q_heads=hq, num_kv_heads=hkv, head_size=d,
                    block_size=bs, causal=True, seed=seed, seqs=seqs,
                    num_blocks=num_blocks, signs=signs, block_table=table,
                    outlier_channels=outliers, outlier_scale=outlier_scale)


def custom_workload(num_q_heads: int, num_kv_heads: int, head_size: int,
                    seqs: List[Tuple[int, int]], seed: int = 7, spare: int = 3,
                    block_size: int = 16, causal: bool = True, sliding_window: int = 0) -> Workload:
    """A workload with explicit shapes, for parity sweeps and edge cases."""
    g = torch.Generator("cpu")
    g.manual_seed(seed)
    signs = (torch.randint(0, 2, (head_size,), generator=g, dtype=torch.int64) * 2 - 1).to(torch.int8)
    nblk = [_blocks(kv, block_size) for _, kv in seqs]
    num_blocks = max(1, sum(nblk) + spare)
    perm = torch.randperm(num_blocks, generator=g).to(torch.int32)
    max_blocks = max([1] + nblk)
    table = torch.full((len(seqs), max_blocks), -1, dtype=torch.int32)
    off = 0
    for s, n in enumerate(nblk):
        table[s, :n] = perm[off:off + n]
        off += n
    return Workload(name="custom", num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                    head_size=head_size, block_size=block_size, causal=causal, seed=seed,
                    seqs=list(seqs), num_blocks=num_blocks, signs=signs, block_table=table,
                    outlier_channels=None, outlier_scale=1.0, sliding_window=sliding_window)


def describe(w: Workload) -> Dict:
    return {
        "workload": w.name,
        "num_q_heads": w.num_q_heads,
        "num_kv_heads": w.num_kv_heads,
        "head_size": w.head_size,
        "block_size": w.block_size,
        "num_seqs": w.num_seqs,
        "num_q_tokens": w.num_q_tokens,
        "sum_kv_len": int(sum(kv for _, kv in w.seqs)),
        "max_seq_len": w.max_seq_len,
        "num_blocks": w.num_blocks,
        "seed": w.seed,
    }
