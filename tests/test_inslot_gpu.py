"""The in-slot scale layout (uint8 [blocks][2][16][Hkv][P], codes then the
f32 scale in every P-byte slot) for both formats, through the C ABI.

The layout only moves bytes, so the in-slot paths must reproduce the
separate-layout paths exactly: writes byte for byte (after the oracle's
to_inslot packing of the separate caches), attention bit for bit on the
same cache contents (same kernels, same schedule).  A write stores a slot's
scale and the padding after it as the slot's last 16 bytes (the scale, then
zeros); the padding of slots no write touched keeps its bytes, and
attention never reads padding (the attention cases fill it with PAD)."""

import math

import numpy as np
import pytest
import torch

from oracle import kvint4_oracle as O
from int4_token_head_gb300 import _lib, synthetic
from int4_token_head_gb300.paged import PagedKV
from tests.helpers import assert_close_attention, oracle_attention, oracle_write_history_and_step

pytestmark = pytest.mark.gpu
PAD = 0xEE


def _written_padding_zeroed(want, slots, cb):
    """The in-slot cache a write leaves: want (built with PAD padding) with
    the padding of every written slot (both halves, every head) zeroed."""
    for s_ in np.asarray(slots):
        if s_ >= 0:
            want[s_ // 16, :, s_ % 16, :, cb + 4:] = 0
    return want


@pytest.mark.parametrize("int8", [False, True])
@pytest.mark.parametrize("d,hkv", [(64, 8), (96, 32), (128, 8), (192, 4), (256, 2), (128, 40)])
def test_inslot_write_matches_separate_write(d, hkv, int8):
    T, nb = 150, 12
    g = torch.Generator().manual_seed(d + hkv + int8)
    k = torch.randn((T, hkv, d), generator=g).to(torch.bfloat16).cuda()
    v = torch.randn((T, hkv, d), generator=g).to(torch.bfloat16).cuda()
    slots = torch.randperm(nb * 16, generator=g)[:T].to(torch.int64)
    slots[3] = -1
    slots = slots.cuda()
    signs = (torch.randint(0, 2, (d,), generator=g) * 2 - 1).to(torch.int8).cuda()
    cb = d if int8 else d // 2
    kc = torch.zeros((nb, 16, hkv, cb), dtype=torch.int8 if int8 else torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    ks = torch.zeros((nb, 16, hkv), dtype=torch.float32, device="cuda")
    vs = torch.zeros_like(ks)
    if int8:
        _lib.write_int8(k, v, slots, kc, vc, ks, vs)
    else:
        _lib.write(k, v, slots, kc, vc, ks, vs, signs)
    # both layouts start from zero codes and scales (the in-slot padding holds PAD)
    ins = torch.from_numpy(O.to_inslot(np.zeros(kc.shape, np.uint8), np.zeros(kc.shape, np.uint8),
                                       np.zeros(ks.shape, np.float32), np.zeros(ks.shape, np.float32),
                                       fill=PAD)).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _lib.write_inslot(k, v, slots, ins, signs=signs, int8=int8, dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    want = O.to_inslot(kc.cpu().numpy(), vc.cpu().numpy(), ks.cpu().numpy(), vs.cpu().numpy(), fill=PAD)
    want = _written_padding_zeroed(want, slots.cpu().numpy(), cb)
    assert np.array_equal(ins.cpu().numpy(), want)


def test_inslot_int8_write_matches_the_oracle():
    d, hkv, T, nb = 128, 4, 90, 8
    g = torch.Generator().manual_seed(77)
    k = torch.randn((T, hkv, d), generator=g).to(torch.bfloat16)
    v = torch.randn((T, hkv, d), generator=g).to(torch.bfloat16)
    slots = torch.randperm(nb * 16, generator=g)[:T].to(torch.int64)
    kc = np.zeros((nb, 16, hkv, d), np.int8)
    vc = kc.copy()
    ks = np.zeros((nb, 16, hkv), np.float32)
    vs = ks.copy()
    O.write_cache_int8(k.double().numpy(), v.double().numpy(), slots.numpy(), kc, vc, ks, vs, 16)
    ins = torch.from_numpy(O.to_inslot(np.zeros_like(kc), np.zeros_like(vc), np.zeros_like(ks), np.zeros_like(vs),
                                       fill=PAD)).cuda()
    _lib.write_inslot(k.cuda(), v.cuda(), slots.cuda(), ins, int8=True)
    torch.cuda.synchronize()
    want = _written_padding_zeroed(O.to_inslot(kc, vc, ks, vs, fill=PAD), slots.numpy(), d)
    assert np.array_equal(ins.cpu().numpy(), want)


ATT_CASES = [
    ("decode_d128_g4", 32, 8, 128, [(1, 300), (1, 37), (1, 1)], True, 0),
    ("decode_d96_g1", 8, 8, 96, [(1, 200), (1, 33)], True, 0),
    ("prefill_d192_g4", 8, 2, 192, [(100, 130), (17, 17)], True, 0),
    ("mixed_window_d128", 16, 4, 128, [(1, 300), (40, 90), (1, 20)], True, 30),
    ("decode_d256_g2", 4, 2, 256, [(1, 77), (1, 160)], True, 0),
]


@pytest.mark.parametrize("int8", [False, True])
@pytest.mark.parametrize("case", ATT_CASES, ids=lambda c: c[0])
def test_inslot_attention_equals_separate_attention(case, int8):
    name, hq, hkv, d, seqs, causal, win = case
    w = synthetic.custom_workload(hq, hkv, d, seqs, seed=41, causal=causal, sliding_window=win)
    pk = PagedKV(w, fmt="int8" if int8 else "int4")
    pk.populate_history(gen_device="cpu")
    q, k, v, slots = pk.step_inputs(gen_device="cpu")
    pk.write(k, v, slots)
    out_sep = torch.full((w.num_q_tokens, hq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    pk.attend(q, out_sep)
    torch.cuda.synchronize()
    ins = torch.from_numpy(O.to_inslot(pk.k_cache.cpu().numpy(), pk.v_cache.cpu().numpy(),
                                       pk.k_scale.cpu().numpy(), pk.v_scale.cpu().numpy(), fill=PAD)).cuda()
    out_ins = torch.full_like(out_sep, float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _lib.attention_inslot(q, ins, pk.block_table, pk.seq_lens, pk.query_start_loc, w.max_query_len,
                          w.max_seq_len, pk.softmax_scale, w.causal, out_ins, pk.workspace, signs=pk.signs,
                          int8=int8, dev_status=status, sliding_window=win)
    torch.cuda.synchronize()
    assert status.item() == 0 and pk.status.item() == 0
    assert torch.equal(out_ins, out_sep), name


def test_inslot_int4_attention_against_the_oracle():
    w = synthetic.custom_workload(16, 4, 192, [(1, 300), (60, 60), (1, 45), (25, 200)], seed=43)
    caches = oracle_write_history_and_step(w)
    ins = torch.from_numpy(O.to_inslot(*caches, fill=PAD)).cuda()
    q = w.queries("cpu")
    out = torch.full((w.num_q_tokens, w.num_q_heads, w.head_size), float("nan"), dtype=torch.bfloat16,
                     device="cuda")
    ws = torch.empty(_lib.attention_workspace_size(w.num_seqs, w.num_q_tokens, w.num_q_heads, w.num_kv_heads,
                                                   w.head_size), dtype=torch.uint8, device="cuda")
    _lib.attention_inslot(q.cuda(), ins, w.block_table.cuda(), w.seq_lens.cuda(), w.query_start_loc.cuda(),
                          w.max_query_len, w.max_seq_len, 1.0 / math.sqrt(w.head_size), w.causal, out, ws,
                          signs=w.signs.cuda())
    torch.cuda.synchronize()
    assert_close_attention(out.float().cpu().numpy(), oracle_attention(w, q, caches), what="in-slot int4")
