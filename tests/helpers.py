"""Shared test helpers: run the oracle on a synthetic workload, compare outputs."""

import math

import numpy as np
import torch

from oracle import kvint4_oracle as O


def np_cache(w):
    return [t.numpy() for t in w.empty_cache("cpu")]


def oracle_write_history_and_step(w, caches=None):
    """Oracle write of every history token and every step token (on CPU)."""
    kc, vc, ks, vs = caches if caches is not None else np_cache(w)
    signs = w.signs.numpy()
    for s, (q, kv) in enumerate(w.seqs):
        k, v = w.seq_kv(s, "cpu")
        O.write_cache(k.float().numpy(), v.float().numpy(), w.slots(s, 0, kv).numpy(), kc, vc, ks, vs,
                      w.block_size, signs)
    return kc, vc, ks, vs


def oracle_attention(w, q, caches, seqs=None, heads=None):
    kc, vc, ks, vs = caches
    qn = q.float().cpu().numpy()
    bt = w.block_table.numpy()
    sl = w.seq_lens.numpy()
    qsl = w.query_start_loc.numpy()
    scale = 1.0 / math.sqrt(w.head_size)
    if seqs is None:
        return O.attention(qn, kc, vc, ks, vs, bt, sl, qsl, w.num_kv_heads, w.block_size, scale, w.causal,
                           w.signs.numpy(), sliding_window=w.sliding_window)
    out = {}
    for s in seqs:
        out[s] = O.attention_seq(qn, kc, vc, ks, vs, bt, sl, qsl, s, w.num_kv_heads, w.block_size, scale,
                                 w.causal, w.signs.numpy(), q_heads=heads, sliding_window=w.sliding_window)
    return out


def corr(a, b):
    a = np.asarray(a, np.float64).ravel()
    b = np.asarray(b, np.float64).ravel()
    return float(np.corrcoef(a, b)[0, 1])


def assert_close_attention(got, ref, atol=5e-2, rtol=5e-2, min_corr=0.9999, what=""):
    """The attention bar: atol = rtol = 5e-2 elementwise and correlation >= 0.9999."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bad = err > atol + rtol * np.abs(ref)
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside atol=rtol={atol}; max abs err {err.max():.4g}"
    c = corr(got, ref)
    assert c >= min_corr, f"{what}: corr {c:.6f} < {min_corr}"
    return float(err.max()), c


def f32_bits(x):
    return np.asarray(x, np.float32).view(np.uint32)


def check_sampled_end_to_end(w, q, out, seqs, heads):
    """End to end on sampled rows: the oracle writes the sampled sequences'
    K/V itself (drawn on the GPU, copied to the host), attends, and every
    sampled (sequence, q head) row of the GPU output must be within atol =
    rtol = 5e-2; the rows together must correlate >= 0.9999 (single 96- or
    128-element rows are too short for a meaningful correlation bar)."""
    qn = q.float().cpu().numpy()
    scale = 1.0 / math.sqrt(w.head_size)
    signs = w.signs.numpy()
    gots, refs = [], []
    for s in seqs:
        ql, L = w.seqs[s]
        k, v = w.seq_kv(s, "cuda")
        k = k.float().cpu().numpy()
        v = v.float().cpu().numpy()
        q0 = int(w.query_start_loc[s])
        for h in heads:
            kvh = h // w.group
            kc, ksc = O.quantize(O.rotate_for_cache(k[:, kvh], signs))
            vc, vsc = O.quantize(O.rotate_for_cache(v[:, kvh], signs))
            k_hat = O.dequantize_original(kc, ksc, signs)
            v_hat = O.dequantize_original(vc, vsc, signs)
            refs.append(O.attention_head(qn[q0:q0 + ql, h], k_hat, v_hat, L - ql, scale, w.causal,
                                         w.sliding_window).ravel())
            gots.append(out[q0:q0 + ql, h].float().cpu().numpy().ravel())
    return assert_close_attention(np.concatenate(gots), np.concatenate(refs),
                                  what=f"{w.name} sampled end to end")


def upload_cache(pk, caches):
    """Copy host (numpy) cache arrays into a PagedKV's device caches."""
    for dst, src in zip((pk.k_cache, pk.v_cache, pk.k_scale, pk.v_scale), caches):
        dst.copy_(torch.from_numpy(src))


def attend_on_oracle_cache(w):
    """The oracle writes the cache; the GPU attends over those same bytes.
    Returns (GPU output, oracle output, device status)."""
    from int4_token_head_gb300.paged import PagedKV
    caches = oracle_write_history_and_step(w)
    pk = PagedKV(w)
    upload_cache(pk, caches)
    q = w.queries("cpu")
    out = torch.full((w.num_q_tokens, w.num_q_heads, w.head_size), float("nan"), dtype=torch.bfloat16,
                     device="cuda")
    pk.attend(q.cuda(), out)
    torch.cuda.synchronize()
    ref = oracle_attention(w, q, caches)
    return out.float().cpu().numpy(), ref, int(pk.status.item())
