"""Parity of kv_int4_attention (CUDA, through the C ABI) with the fp64 oracle.

Two kinds of comparison:
* attention alone: the oracle writes the cache from the synthetic K/V; the
  same bytes are uploaded and both sides attend over them;
* end to end: each side writes its own cache from the same K/V and attends
  (codes may differ by one between the two writes).
The bar is the pages' attention tolerance, atol = rtol = 5e-2, plus
correlation >= 0.9999.
"""

import math

import numpy as np
import pytest
import torch

from oracle import kvint4_oracle as O
from int4_token_head_gb300 import _lib, synthetic
from int4_token_head_gb300.paged import PagedKV
from tests.helpers import (assert_close_attention, attend_on_oracle_cache, corr, oracle_attention,
                           oracle_write_history_and_step, upload_cache)

pytestmark = pytest.mark.gpu


_upload = upload_cache
_attend_on_oracle_cache = attend_on_oracle_cache


CASES = [
    # (name, Hq, Hkv, d, [(q_len, kv_len), ...], causal)
    ("decode_d128_g4", 32, 8, 128, [(1, 37), (1, 300), (1, 16), (1, 1), (1, 129)], True),
    ("decode_d96_g1_phi3", 8, 8, 96, [(1, 200), (1, 33), (1, 64)], True),
    ("decode_d192_g4", 16, 4, 192, [(1, 500), (1, 17)], True),
    ("decode_d64_g8", 16, 2, 64, [(1, 90), (1, 250)], True),
    ("decode_d256_g2", 4, 2, 256, [(1, 77), (1, 160)], True),
    ("decode_d64_four_heads_per_cta", 16, 4, 64, [(1, 90), (1, 250), (1, 7)], True),
    ("decode_d256_four_heads_per_cta", 8, 4, 256, [(1, 77), (1, 160)], True),
    ("decode_d96_spec_q2", 8, 8, 96, [(2, 70), (1, 33)], True),
    ("spec_q2_g4_decode_path", 8, 2, 128, [(2, 50), (2, 2), (1, 40)], True),
    ("q3_g4_prefill_path", 8, 2, 128, [(3, 50), (3, 3)], True),
    ("prefill_d128_g4", 16, 4, 128, [(40, 40), (70, 100), (5, 5)], True),
    ("prefill_d96_g1", 4, 4, 96, [(33, 33), (20, 90)], True),
    ("prefill_d192_g4", 8, 2, 192, [(100, 130), (17, 17)], True),
    ("prefill_d64_g16", 32, 2, 64, [(9, 20), (3, 40)], True),
    ("prefill_d256_g1", 2, 2, 256, [(30, 64), (16, 16)], True),
    ("mixed_any_order", 16, 4, 192, [(1, 300), (60, 60), (1, 45), (25, 200), (1, 1)], True),
    ("noncausal_prefill", 8, 2, 128, [(20, 60), (7, 7)], False),
    ("decode_g16_prefill_kernel", 32, 2, 128, [(1, 100), (1, 33)], True),
    # decode lanes: head-group counts that are not powers of two (3 groups of
    # four heads, 7 groups of one), and more groups than CTAs, where each lane
    # walks several groups (609 groups of four heads: 203 lanes of 3)
    ("decode_three_head_groups", 12, 12, 128, [(1, 90), (1, 300), (1, 5)], True),
    ("decode_seven_head_groups", 14, 7, 64, [(1, 120), (1, 33)], True),
    ("decode_groups_beyond_grid", 2436, 2436, 64, [(1, 20), (1, 37)], True),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_attention_on_oracle_cache(case):
    name, hq, hkv, d, seqs, causal = case
    w = synthetic.custom_workload(hq, hkv, d, seqs, seed=11, causal=causal)
    got, ref, status = _attend_on_oracle_cache(w)
    assert status == 0
    assert_close_attention(got, ref, what=name)


WINDOW_CASES = [
    # (name, Hq, Hkv, d, [(q_len, kv_len), ...], causal, sliding_window)
    ("win64_decode_d128_g4", 32, 8, 128, [(1, 300), (1, 37), (1, 16), (1, 1), (1, 129)], True, 64),
    ("win37_decode_d96_g1", 8, 8, 96, [(1, 200), (1, 33), (1, 64)], True, 37),
    ("win1_decode_d128_g4", 16, 4, 128, [(1, 90), (1, 5)], True, 1),
    ("win_ge_len_decode_d192", 16, 4, 192, [(1, 500), (1, 17)], True, 1000),
    ("win5_spec_q2_decode_path", 8, 2, 128, [(2, 50), (2, 2), (1, 40)], True, 5),
    ("win24_prefill_d128_g4", 16, 4, 128, [(40, 40), (70, 100), (5, 5)], True, 24),
    ("win100_prefill_d64_g16", 32, 2, 64, [(130, 300), (3, 40)], True, 100),
    ("win50_mixed_d192", 16, 4, 192, [(1, 300), (60, 60), (1, 45), (25, 200), (1, 1)], True, 50),
    ("win10_noncausal_prefill", 8, 2, 128, [(20, 60), (7, 7)], False, 10),
    ("win20_decode_g16_prefill_kernel", 32, 2, 128, [(1, 100), (1, 33)], True, 20),
]


@pytest.mark.parametrize("case", WINDOW_CASES, ids=lambda c: c[0])
def test_attention_sliding_window_on_oracle_cache(case):
    name, hq, hkv, d, seqs, causal, win = case
    w = synthetic.custom_workload(hq, hkv, d, seqs, seed=13, causal=causal, sliding_window=win)
    got, ref, status = _attend_on_oracle_cache(w)
    assert status == 0
    assert_close_attention(got, ref, what=name)


def test_sliding_window_blocks_before_the_window_are_never_read():
    """Blocks wholly before every query's window may hold anything (here
    NaN-payload scales and garbage codes): the output must not change."""
    w = synthetic.custom_workload(16, 4, 128, [(1, 400), (3, 260)], seed=17, sliding_window=48)
    caches = oracle_write_history_and_step(w)
    pk = PagedKV(w)
    _upload(pk, caches)
    q = w.queries("cpu").cuda()
    out_a = torch.empty((w.num_q_tokens, w.num_q_heads, w.head_size), dtype=torch.bfloat16, device="cuda")
    pk.attend(q, out_a)
    for s, (ql, L) in enumerate(w.seqs):
        first = (L - ql - 48 + 1) // 16
        for blk in w.block_table[s, :max(0, first)].tolist():
            pk.k_cache[blk].fill_(0x77)
            pk.v_cache[blk].fill_(0x77)
            pk.k_scale[blk].fill_(float("nan"))
            pk.v_scale[blk].fill_(float("nan"))
    out_b = torch.empty_like(out_a)
    pk.attend(q, out_b)
    torch.cuda.synchronize()
    assert pk.status.item() == 0
    assert torch.equal(out_a, out_b)


@pytest.mark.parametrize("name", ["tiny"])
def test_attention_tiny_end_to_end(name):
    w = synthetic.make_workload(name)
    pk = PagedKV(w)
    pk.populate_history(gen_device="cpu")
    q, k, v, slots = pk.step_inputs(gen_device="cpu")
    out = torch.full((w.num_q_tokens, w.num_q_heads, w.head_size), float("nan"), dtype=torch.bfloat16,
                     device="cuda")
    pk.step(q, k, v, slots, out)
    torch.cuda.synchronize()
    assert pk.status.item() == 0
    ref = oracle_attention(w, q, oracle_write_history_and_step(w))
    assert_close_attention(out.float().cpu().numpy(), ref, what=name)


def test_attention_200_seed_sweep_tiny():
    """The pages' seed-sweep probe on the INT4 attention test shape (block
    16, head 128, seqs (4,128),(4,97)): 0/200 seeds fail atol=rtol=5e-2, and
    correlation stays at 1.0000 (reported worst abs diffs were 0.006-0.021)."""
    worst = 0.0
    fails = 0
    min_corr = 1.0
    for seed in range(200):
        w = synthetic.make_workload("tiny", seed=5000 + seed)
        got, ref, status = _attend_on_oracle_cache(w)
        assert status == 0
        err = np.abs(got - ref)
        worst = max(worst, float(err.max()))
        fails += int((err > 5e-2 + 5e-2 * np.abs(ref)).any())
        min_corr = min(min_corr, corr(got, ref))
    assert fails == 0
    assert min_corr >= 0.9999
    assert worst <= 0.021


def test_unwritten_slots_never_read():
    """Caches keep NaN-payload scales in every unwritten slot; any unmasked
    read past seq_len or into a spare block would poison the output."""
    w = synthetic.custom_workload(8, 2, 128, [(1, 17), (5, 21), (1, 3)], seed=3, spare=5)
    got, ref, status = _attend_on_oracle_cache(w)
    assert np.isfinite(got).all()
    assert_close_attention(got, ref, what="nan-sentinel")


def test_bad_block_and_bad_sequence_are_reported_not_trapped():
    w = synthetic.custom_workload(8, 2, 128, [(1, 40), (2, 1), (1, 20)], seed=4)
    # seq 1 claims q_len 2 > seq_len 1: invalid, skipped
    caches = [t.numpy() for t in w.empty_cache("cpu")]
    pk = PagedKV(w)
    _upload(pk, caches)
    pk.block_table[2, 0] = w.num_blocks + 7  # out of range block for seq 2
    q = w.queries("cuda")
    out = torch.zeros((w.num_q_tokens, w.num_q_heads, w.head_size), dtype=torch.bfloat16, device="cuda")
    out[1:3] = 7.0
    pk.attend(q, out)
    torch.cuda.synchronize()
    st = pk.status.item()
    assert st & _lib.DEV_BAD_SEQ and st & _lib.DEV_BAD_BLOCK
    assert torch.all(out[1:3] == 7.0)  # rows of the invalid sequence untouched


def test_sequences_without_queries_and_an_empty_batch():
    """Sequences with q_len = 0 (one of them with no keys at all) contribute
    no rows and leave the other sequences' rows exact; a batch with no
    sequences (or no query tokens) enqueues nothing and returns OK."""
    w = synthetic.custom_workload(8, 2, 128, [(0, 50), (1, 40), (0, 0), (3, 30), (0, 17)], seed=23)
    got, ref, status = attend_on_oracle_cache(w)
    assert status == 0
    assert_close_attention(got, ref, what="sequences without queries")
    pk = PagedKV(w)
    q = torch.empty((0, 8, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    none = torch.empty((0,), dtype=torch.int32, device="cuda")
    _lib.attention(q, pk.k_cache, pk.v_cache, pk.k_scale, pk.v_scale, pk.block_table[:0], none,
                   torch.zeros(1, dtype=torch.int32, device="cuda"), 0, 0, pk.softmax_scale, True, pk.signs, out,
                   pk.workspace, dev_status=pk.status)
    torch.cuda.synchronize()
    assert pk.status.item() == 0


@pytest.mark.parametrize("hq,hkv", [(8, 2), (4, 2)])
def test_understated_max_query_len_is_reported_not_dropped(hq, hkv):
    """max_query_len sizes the launches (decode columns, whether a prefill
    launch is made, the reduce segments): a sequence whose q_len exceeds it
    is invalid metadata, so it is skipped with KV_INT4_DEV_BAD_SEQ and its
    rows stay untouched, while the other sequences are still correct."""
    w = synthetic.custom_workload(hq, hkv, 128, [(1, 40), (2, 30), (1, 20)], seed=19)
    caches = oracle_write_history_and_step(w)
    pk = PagedKV(w)
    _upload(pk, caches)
    q = w.queries("cpu")
    out = torch.full((w.num_q_tokens, hq, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    _lib.attention(q.cuda(), pk.k_cache, pk.v_cache, pk.k_scale, pk.v_scale, pk.block_table, pk.seq_lens,
                   pk.query_start_loc, 1, w.max_seq_len, pk.softmax_scale, w.causal, pk.signs, out, pk.workspace,
                   dev_status=pk.status)
    torch.cuda.synchronize()
    assert pk.status.item() & _lib.DEV_BAD_SEQ
    assert torch.all(out[1:3] == 7.0)  # sequence 1's two query rows
    ref = oracle_attention(w, q, caches)
    got = out.float().cpu().numpy()
    keep = [0, 3]
    assert_close_attention(got[keep], ref[keep], what="sequences within max_query_len")


def _magnitude_kv(w, s, vmul_big):
    """K/V of sequence s with per-block magnitudes: V x vmul_big in blocks 6
    and 11 (V scales near 3000, far above 128), K x 3.5 in block 6 (the row
    max rises by 4 to 8 log2 units there, where P' = p * v_scale would
    overflow f16 unless the reference follows the max) and K x 10 in block 9
    (a jump of more than 8 log2 units)."""
    k, v = w.seq_kv(s, "cpu")
    k, v = k.float(), v.float()
    kv = k.shape[0]
    blk = torch.arange(kv) // w.block_size
    vmul = torch.where((blk == 6) | (blk == 11), vmul_big, 1.0)
    kmul = torch.ones(kv)
    kmul[blk == 6] = 3.5
    kmul[blk == 9] = 10.0
    return (k * kmul[:, None, None]).to(torch.bfloat16), (v * vmul[:, None, None]).to(torch.bfloat16)


@pytest.mark.parametrize("fmt", ["int4", "int8"])
@pytest.mark.parametrize("d", [128, 192])
def test_prefill_rescale_policies_with_large_v_scales_and_score_jumps(fmt, d):
    """The tensor-core prefill moves a row's exponent reference lazily only
    while every V scale of the step is below 128; this case mixes steps of
    both kinds with score jumps below and above the lazy threshold.  Rows
    are compared relative to their own magnitude (max |ref| of the row, at
    least 1)."""
    w = synthetic.custom_workload(16, 4, d, [(150, 150), (64, 230), (1, 200)], seed=53)
    pk = PagedKV(w, fmt=fmt)
    caches = [t.cpu().numpy() for t in (pk.k_cache, pk.v_cache, pk.k_scale, pk.v_scale)]
    vmul_big = 680.0 if fmt == "int4" else 1.27e5  # rotated INT4 scales ~ 4.4 sigma, int8 ~ sigma / 42
    for s, (q, kv) in enumerate(w.seqs):
        k, v = _magnitude_kv(w, s, vmul_big)
        args = (k.double().numpy(), v.double().numpy(), w.slots(s, 0, kv).numpy(), *caches, w.block_size)
        if fmt == "int4":
            O.write_cache(*args, w.signs.numpy())
        else:
            O.write_cache_int8(*args)
    _upload(pk, caches)
    vs = caches[3][np.isfinite(caches[3])]
    assert vs.max() > 1000 and np.median(vs) < 128
    q = w.queries("cpu")
    out = torch.full((w.num_q_tokens, w.num_q_heads, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    pk.attend(q.cuda(), out)
    torch.cuda.synchronize()
    assert pk.status.item() == 0
    args = (q.float().numpy(), *caches, w.block_table.numpy(), w.seq_lens.numpy(), w.query_start_loc.numpy(),
            w.num_kv_heads, w.block_size, 1.0 / math.sqrt(d), w.causal)
    ref = O.attention(*args, w.signs.numpy()) if fmt == "int4" else O.attention_int8(*args)
    scale = np.maximum(1.0, np.abs(ref).max(axis=-1, keepdims=True))
    assert scale.max() > 100  # the large-V blocks carry weight
    assert_close_attention(out.float().cpu().numpy() / scale, ref / scale, what=f"{fmt} d={d} magnitudes")


@pytest.mark.parametrize("fmt", ["int4", "int8"])
@pytest.mark.parametrize("case", [
    ("mixed_window_d128", 16, 4, 128, [(1, 300), (40, 90), (1, 20)], 30),
    ("mixed_d128", 16, 4, 128, [(1, 300), (40, 90), (1, 20)], 0),
    ("prefill_d192_g4", 8, 2, 192, [(100, 130), (17, 17)], 0),
    ("prefill_d96_g1_window", 4, 4, 96, [(70, 200), (33, 33)], 50),
], ids=lambda c: c[0] if isinstance(c, tuple) else c)
def test_attention_is_deterministic(case, fmt):
    """Repeated calls on the same cache give bit-identical outputs: the
    schedule's order (atomic item counter, stream-K ranges) and the prefill's
    pipeline timing must not change any rounding."""
    name, hq, hkv, d, seqs, win = case
    w = synthetic.custom_workload(hq, hkv, d, seqs, seed=41, causal=True, sliding_window=win)
    pk = PagedKV(w, fmt=fmt)
    pk.populate_history(gen_device="cpu")
    q, k, v, slots = pk.step_inputs(gen_device="cpu")
    pk.write(k, v, slots)
    first = None
    for _ in range(6):
        out = torch.full((w.num_q_tokens, hq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
        pk.attend(q, out)
        torch.cuda.synchronize()
        if first is None:
            first = out.clone()
        else:
            assert torch.equal(out, first), name
    assert pk.status.item() == 0


@pytest.mark.parametrize("fmt", ["int4", "int8"])
@pytest.mark.parametrize("d", [64, 96, 128, 192, 256])
def test_strided_offset_q_and_out_match_contiguous(d, fmt):
    """q and out as views with a token stride of Hq*d + 24 elements and a
    start 16 bytes past a 256-byte boundary (legal: 16-byte aligned, stride a
    multiple of 8; neither is 32-byte aligned) give the bit-identical output
    of contiguous tensors, through prefill, decode and reduce, and write
    nothing between the rows."""
    seqs = [(150, 150), (1, 700), (37, 300), (1, 1500), (64, 64), (2, 90)]
    w = synthetic.custom_workload(16, 4, d, seqs, seed=31)
    pk = PagedKV(w, fmt=fmt)
    pk.populate_history()
    q, k_new, v_new, slots = pk.step_inputs()
    pk.write(k_new, v_new, slots)
    T, hq = w.num_q_tokens, w.num_q_heads
    ref = torch.empty((T, hq, d), dtype=torch.bfloat16, device="cuda")
    pk.attend(q, ref)
    row, off = hq * d + 24, 8
    qbuf = torch.zeros(off + T * row, dtype=torch.bfloat16, device="cuda")
    qv = torch.as_strided(qbuf, (T, hq, d), (row, d, 1), storage_offset=off)
    qv.copy_(q)
    sentinel = torch.tensor(-12345.0, dtype=torch.bfloat16)
    obuf = torch.full((off + T * row,), float(sentinel), dtype=torch.bfloat16, device="cuda")
    ov = torch.as_strided(obuf, (T, hq, d), (row, d, 1), storage_offset=off)
    pk.attend(qv, ov)
    torch.cuda.synchronize()
    assert int(pk.status.item()) == 0
    assert torch.equal(ov.contiguous().view(torch.int16), ref.view(torch.int16))
    written = torch.zeros(off + T * row, dtype=torch.bool, device="cuda")
    torch.as_strided(written, (T, hq, d), (row, d, 1), storage_offset=off).fill_(True)
    assert torch.all(obuf[~written] == sentinel)
