"""A seeded randomized sweep of attention shapes, GPU against the oracle.

Each case draws a head size, a kv-head count and group size, a batch of
sequences (mostly single-token decodes, some speculative and prefill
lengths, from one key up to a few hundred), causality and a sliding window;
the oracle writes the cache and the GPU attends over those same bytes.  The
bar is the pages' attention tolerance ("Rotate KV into RHT domain in the
INT4 unified attn test", Claims / Tolerance: atol = rtol = 5e-2) and
correlation >= 0.9999.  The draws come from fixed seeds, so the sweep is
the same on every run; each case's shape is in its test id."""

import random

import pytest

from int4_token_head_gb300 import synthetic
from tests.helpers import assert_close_attention, attend_on_oracle_cache

pytestmark = pytest.mark.gpu

N_CASES = 100


def _draw(i):
    r = random.Random(9000 + i)
    d = r.choice([64, 96, 128, 192, 256])
    hkv = r.choice([1, 2, 3, 4, 5, 6, 8])
    g = r.choice([1, 2, 4, 8])
    seqs = []
    for _ in range(r.randint(1, 10)):
        u = r.random()
        q = 1 if u < 0.6 else r.choice([2, 3]) if u < 0.75 else r.randint(4, 80)
        seqs.append((q, q + r.choice([0, r.randint(1, 15), r.randint(16, 120), r.randint(121, 400)])))
    causal = r.random() < 0.85
    window = r.choice([0, 0, 0, 1, 17, 64, 300])
    return d, hkv, g, seqs, causal, window


def _case_id(i):
    d, hkv, g, seqs, causal, window = _draw(i)
    return f"{i}-d{d}-hkv{hkv}-g{g}-n{len(seqs)}-{'c' if causal else 'nc'}-w{window}"


@pytest.mark.parametrize("i", range(N_CASES), ids=_case_id)
def test_random_shapes_on_oracle_cache(i):
    d, hkv, g, seqs, causal, window = _draw(i)
    w = synthetic.custom_workload(hkv * g, hkv, d, seqs, seed=500 + i, causal=causal, sliding_window=window)
    got, ref, status = attend_on_oracle_cache(w)
    assert status == 0
    assert_close_attention(got, ref, what=_case_id(i))


# ---------------------------------------------------------------------------
# the write, randomized: head size, kv heads (up to 40, past the tensor-core
# kernel's tile), token count, slot pattern (padding tokens, a sparse cache)
# and value ranges; the prerotated hook must match the oracle bit for bit,
# the full write within one code (the GPU rotates in fp32, the oracle in fp64)
# ---------------------------------------------------------------------------
N_WRITE_CASES = 40


def _draw_write(i):
    r = random.Random(7000 + i)
    d = r.choice([64, 96, 128, 192, 256])
    hkv = r.choice([1, 2, 3, 4, 8, 16, 33, 40])
    T = r.choice([1, r.randint(2, 64), r.randint(65, 600), r.randint(601, 3000)])
    nb = (T + 15) // 16 + r.choice([0, 1, 7, 100])
    return d, hkv, T, nb


def _write_case_id(i):
    d, hkv, T, nb = _draw_write(i)
    return f"{i}-d{d}-hkv{hkv}-T{T}-nb{nb}"


def _write_inputs(i):
    import numpy as np
    import torch
    d, hkv, T, nb = _draw_write(i)
    g = torch.Generator().manual_seed(3000 + i)
    # per-vector magnitudes over many binades, some all-zero vectors
    mag = torch.exp2(torch.randint(-30, 30, (T, hkv, 1), generator=g).double())
    k = (torch.randn((T, hkv, d), generator=g, dtype=torch.float64) * mag).to(torch.bfloat16)
    v = (torch.randn((T, hkv, d), generator=g, dtype=torch.float64) * mag.flip(0)).to(torch.bfloat16)
    k[torch.rand((T, hkv), generator=g) < 0.02] = 0
    slots = torch.randperm(nb * 16, generator=g)[:T].to(torch.int64)
    slots[torch.rand(T, generator=g) < 0.05] = -1
    signs = (torch.randint(0, 2, (d,), generator=g) * 2 - 1).to(torch.int8)
    return d, hkv, T, nb, k, v, slots, signs


def _caches(nb, hkv, d, dev):
    w = synthetic.custom_workload(hkv, hkv, d, [(1, 1)])
    w.num_blocks = nb
    return w.empty_cache(dev)


@pytest.mark.parametrize("i", range(N_WRITE_CASES), ids=_write_case_id)
def test_random_writes_against_the_oracle(i):
    import numpy as np
    import torch
    from oracle import kvint4_oracle as O
    from int4_token_head_gb300 import _lib
    from tests.helpers import f32_bits
    d, hkv, T, nb, k, v, slots, signs = _write_inputs(i)

    def gpu(kk, vv, prerotated):
        caches = _caches(nb, hkv, d, "cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        _lib.write(kk.cuda(), vv.cuda(), slots.cuda(), *caches, signs.cuda(), dev_status=status,
                   prerotated=prerotated)
        torch.cuda.synchronize()
        assert status.item() == 0
        return [t.cpu().numpy() for t in caches]

    def oracle(kk, vv, prerotated):
        caches = [t.numpy() for t in _caches(nb, hkv, d, "cpu")]
        O.write_cache(kk.double().numpy(), vv.double().numpy(), slots.numpy(), *caches, 16,
                      signs.numpy(), prerotated=prerotated)
        return caches

    # prerotated: the oracle's own bf16 rotation of the inputs, then bit for bit
    sg = signs.numpy().astype(np.float64)
    ky = torch.from_numpy(O.rotate_for_cache(k.double().numpy(), sg)).to(torch.bfloat16)
    vy = torch.from_numpy(O.rotate_for_cache(v.double().numpy(), sg)).to(torch.bfloat16)
    for a, b in zip(gpu(ky, vy, True), oracle(ky, vy, True)):
        assert np.array_equal(f32_bits(a), f32_bits(b)) if a.dtype == np.float32 else np.array_equal(a, b)

    # the full write: untouched slots bit for bit, codes within one
    got, ref = gpu(k, v, False), oracle(k, v, False)
    written = np.zeros(nb * 16, bool)
    written[slots[slots >= 0].numpy()] = True
    written = written.reshape(nb, 16)
    for which in (0, 1):
        assert np.array_equal(got[which][~written], ref[which][~written])
        assert np.array_equal(f32_bits(got[2 + which][~written]), f32_bits(ref[2 + which][~written]))
        diff = np.abs(O.unpack_codes(got[which][written]).astype(np.int32) -
                      O.unpack_codes(ref[which][written]).astype(np.int32))
        assert diff.max(initial=0) <= 1
        gs, rs = got[2 + which][written].astype(np.float64), ref[2 + which][written].astype(np.float64)
        nz = rs > 0
        assert np.array_equal(gs[~nz], rs[~nz])  # zero vectors: scale 0 on both sides
        if nz.any():
            assert (np.abs(gs[nz] - rs[nz]) / rs[nz]).max() <= 2.0 ** -7
