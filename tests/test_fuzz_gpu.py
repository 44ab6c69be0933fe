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
