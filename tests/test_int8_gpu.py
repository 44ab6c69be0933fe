"""Parity of the int8_per_token_head sibling mode (kv_int8_write and
kv_int8_attention, CUDA through the C ABI) with the fp64 oracle
(quantize_int8 / write_cache_int8 / attention_int8).

The write has no rotation, so codes and scales must match the oracle bit
for bit; attention is held to the pages' bar (atol = rtol = 5e-2,
correlation >= 0.9999) on the oracle's cache."""

import math

import numpy as np
import pytest
import torch

from oracle import kvint4_oracle as O
from int4_token_head_gb300 import _lib, synthetic
from tests.helpers import assert_close_attention, corr, f32_bits

pytestmark = pytest.mark.gpu
HEADS = [64, 96, 128, 192, 256]
SENT_CODE = -91  # 0xA5
SENT_SCALE_BITS = 0x7FC00A5A


def _caches(nb, hkv, d, device):
    kc = torch.full((nb, 16, hkv, d), SENT_CODE, dtype=torch.int8, device=device)
    vc = kc.clone()
    ks = torch.full((nb, 16, hkv), SENT_SCALE_BITS, dtype=torch.int32, device=device).view(torch.float32)
    return kc, vc, ks, ks.clone()


def _values(T, hkv, d, seed):
    """bf16 K/V with magnitudes over many binades plus special vectors."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((T, hkv, d), generator=g) * torch.exp(torch.empty((T, hkv, 1)).uniform_(-8, 8, generator=g))
    x = x.to(torch.bfloat16)
    x[0, 0] = 0                                              # zero vector
    x[1, 0] = (torch.randn(d, generator=g) * 2.0 ** -124).to(torch.bfloat16)  # absmax below 2^-119: flushed
    tie = torch.tensor([(i % 255) - 127 + (0.5 if i % 3 == 0 else 0.0) for i in range(d)]).clamp(-126.5, 126.5)
    tie[5] = 127.0
    x[2, 0] = tie.to(torch.bfloat16)                         # s = 1: exact ties to even
    return x


def _gpu_write(k, v, slots, nb):
    hkv, d = k.shape[1], k.shape[2]
    kc, vc, ks, vs = _caches(nb, hkv, d, "cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _lib.write_int8(k.cuda(), v.cuda(), slots.cuda(), kc, vc, ks, vs, dev_status=status)
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in (kc, vc, ks, vs)], int(status.item())


def _oracle_write(k, v, slots, nb):
    hkv, d = k.shape[1], k.shape[2]
    caches = [t.numpy() for t in _caches(nb, hkv, d, "cpu")]
    bad = O.write_cache_int8(k.double().numpy(), v.double().numpy(), slots.numpy(), *caches, 16)
    return caches, bad


def _assert_caches_equal(got, ref):
    for a, b, name in zip(got, ref, ["k_cache", "v_cache", "k_scale", "v_scale"]):
        if a.dtype == np.float32:
            assert np.array_equal(f32_bits(a), f32_bits(b)), name
        else:
            assert np.array_equal(a, b), name


@pytest.mark.parametrize("d", HEADS)
@pytest.mark.parametrize("hkv", [1, 3, 8])
def test_int8_write_bit_exact(d, hkv):
    T, nb = 213, 20  # ragged against every warp step
    k = _values(T, hkv, d, 10 * d + hkv)
    v = _values(T, hkv, d, 20 * d + hkv)
    g = torch.Generator().manual_seed(d + hkv)
    slots = torch.randperm(nb * 16, generator=g)[:T].to(torch.int64)
    slots[7] = -1
    got, status = _gpu_write(k, v, slots, nb)
    ref, bad = _oracle_write(k, v, slots, nb)
    assert status == 0 and bad == []
    _assert_caches_equal(got, ref)


@pytest.mark.parametrize("d", [64, 128, 192])
def test_int8_write_scale_exact_over_all_absmax_mantissas(d):
    """Single-nonzero vectors: absmax is |c| itself, the scale must be
    fp32(|c| / 127) bit for bit (codes +-127) while c sweeps all 128 bf16
    mantissas over exponents from below the flush bound (2^-119) to 2^126."""
    hkv = 4
    exps = [-120, -119, -118, -100, -30, -1, 0, 1, 7, 40, 100, 126]
    vals = np.array([(1 + m / 128) * 2.0 ** e * (1 if (m + e) % 2 else -1) for e in exps for m in range(128)])
    n = len(vals)
    T = (n + hkv - 1) // hkv
    k = torch.zeros((T, hkv, d), dtype=torch.float64)
    v = torch.zeros((T, hkv, d), dtype=torch.float64)
    for u in range(T * hkv):
        t, h = divmod(u, hkv)
        k[t, h, (7 * u + 3) % d] = float(vals[u % n])
        v[t, h, (5 * u + 1) % d] = float(vals[(3 * u + 11) % n])
    k, v = k.to(torch.bfloat16), v.to(torch.bfloat16)
    nb = (T + 15) // 16 + 2
    slots = torch.randperm(nb * 16, generator=torch.Generator().manual_seed(d))[:T].to(torch.int64)
    got, status = _gpu_write(k, v, slots, nb)
    ref, _ = _oracle_write(k, v, slots, nb)
    assert status == 0
    _assert_caches_equal(got, ref)


def test_int8_write_bad_slot_reported_and_zero_tokens():
    d, hkv, nb = 128, 2, 4
    k = _values(20, hkv, d, 5)
    slots = torch.arange(20, dtype=torch.int64)
    slots[3] = nb * 16 + 5  # out of range: skipped and reported
    got, status = _gpu_write(k, k, slots, nb)
    assert status & _lib.DEV_BAD_SLOT
    ref, bad = _oracle_write(k, k, slots, nb)
    assert bad == [nb * 16 + 5]
    _assert_caches_equal(got, ref)
    kc, vc, ks, vs = _caches(nb, hkv, d, "cuda")
    empty = torch.empty((0, hkv, d), dtype=torch.bfloat16, device="cuda")
    _lib.write_int8(empty, empty, torch.empty(0, dtype=torch.int64, device="cuda"), kc, vc, ks, vs)
    torch.cuda.synchronize()
    assert torch.all(kc == SENT_CODE)


def _oracle_cache(w):
    kc, vc, ks, vs = [t.numpy() for t in _caches(w.num_blocks, w.num_kv_heads, w.head_size, "cpu")]
    for s, (q, kv) in enumerate(w.seqs):
        k, v = w.seq_kv(s, "cpu")
        O.write_cache_int8(k.double().numpy(), v.double().numpy(), w.slots(s, 0, kv).numpy(), kc, vc, ks, vs, 16)
    return kc, vc, ks, vs


def _gpu_attend(w, caches, q):
    kc, vc, ks, vs = [torch.from_numpy(c).cuda() for c in caches]
    out = torch.full((w.num_q_tokens, w.num_q_heads, w.head_size), float("nan"), dtype=torch.bfloat16,
                     device="cuda")
    ws = torch.empty(_lib.attention_workspace_size(w.num_seqs, w.num_q_tokens, w.num_q_heads, w.num_kv_heads,
                                                   w.head_size), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _lib.attention_int8(q.cuda(), kc, vc, ks, vs, w.block_table.cuda(), w.seq_lens.cuda(),
                        w.query_start_loc.cuda(), w.max_query_len, w.max_seq_len, 1.0 / math.sqrt(w.head_size),
                        w.causal, out, ws, dev_status=status, sliding_window=w.sliding_window)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), int(status.item())


def _oracle_attend(w, caches, q):
    return O.attention_int8(q.float().numpy(), *caches, w.block_table.numpy(), w.seq_lens.numpy(),
                            w.query_start_loc.numpy(), w.num_kv_heads, 16, 1.0 / math.sqrt(w.head_size), w.causal,
                            sliding_window=w.sliding_window)


CASES = [
    # (name, Hq, Hkv, d, [(q_len, kv_len), ...], causal, window)
    ("decode_d128_g4_paired", 32, 8, 128, [(1, 37), (1, 300), (1, 16), (1, 1), (1, 129)], True, 0),
    ("decode_d96_g1", 8, 8, 96, [(1, 200), (1, 33), (1, 64)], True, 0),
    ("decode_d192_g4", 16, 4, 192, [(1, 500), (1, 17)], True, 0),
    ("decode_d64_g8_unpaired", 16, 2, 64, [(1, 90), (1, 250)], True, 0),
    ("decode_d256_g2_hg_capped", 16, 8, 256, [(1, 77), (1, 160)], True, 0),
    ("spec_q2_g4", 8, 2, 128, [(2, 50), (2, 2), (1, 40)], True, 0),
    ("prefill_d128_g4", 16, 4, 128, [(40, 40), (70, 100), (5, 5)], True, 0),
    ("prefill_d96_g1", 4, 4, 96, [(33, 33), (20, 90)], True, 0),
    ("prefill_d256_g1", 2, 2, 256, [(30, 64), (16, 16)], True, 0),
    ("mixed_d192", 16, 4, 192, [(1, 300), (60, 60), (1, 45), (25, 200), (1, 1)], True, 0),
    ("noncausal_prefill", 8, 2, 128, [(20, 60), (7, 7)], False, 0),
    ("window40_mixed", 16, 4, 128, [(1, 300), (30, 90), (1, 20)], True, 40),
    ("decode_g16_prefill_kernel", 32, 2, 128, [(1, 100), (1, 33)], True, 0),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_int8_attention_on_oracle_cache(case):
    name, hq, hkv, d, seqs, causal, win = case
    w = synthetic.custom_workload(hq, hkv, d, seqs, seed=31, causal=causal, sliding_window=win)
    caches = _oracle_cache(w)
    q = w.queries("cpu")
    got, status = _gpu_attend(w, caches, q)
    assert status == 0
    assert_close_attention(got, _oracle_attend(w, caches, q), what=name)


def test_int8_end_to_end_write_then_attend():
    """GPU write + GPU attention against oracle write + oracle attention: the
    two caches are bit-identical, so the outputs meet the same bar."""
    w = synthetic.custom_workload(32, 8, 128, [(1, 700), (1, 1500), (4, 300)], seed=33)
    kc, vc, ks, vs = _caches(w.num_blocks, 8, 128, "cuda")
    for s, (q, kv) in enumerate(w.seqs):
        k, v = w.seq_kv(s, "cpu")  # the same draws as the oracle's
        _lib.write_int8(k.cuda(), v.cuda(), w.slots(s, 0, kv).cuda(), kc, vc, ks, vs)
    torch.cuda.synchronize()
    ref_caches = _oracle_cache(w)
    _assert_caches_equal([t.cpu().numpy() for t in (kc, vc, ks, vs)], ref_caches)
    q = w.queries("cpu")
    got, status = _gpu_attend(w, [t.cpu().numpy() for t in (kc, vc, ks, vs)], q)
    ref = _oracle_attend(w, ref_caches, q)
    assert status == 0
    assert_close_attention(got, ref, what="int8 end to end")
    assert corr(got, ref) >= 0.9999
