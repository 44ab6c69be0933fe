"""Full-size parity of the named workloads, on the whole output, in the
bench's launch configuration.

For each workload the GPU writes every history token and the step's new
tokens through kv_int4_write, then attends through kv_int4_attention.  Then:

* attention alone, every output row: the GPU-written caches are dumped to
  files, and the fp64 oracle recomputes attention over those same cache
  bytes for every (sequence, q head), in a spawn process pool over the host
  cores.  The bar is the pages' attention tolerance ("Rotate KV into RHT
  domain in the INT4 unified attn test", Claims / Tolerance: atol = rtol =
  5e-2) on every element, and correlation >= 0.9999 over the whole output
  and over every (token, q head) row on its own;
* the write, code by code: the oracle quantises the same K/V (drawn on the
  GPU, copied to the host) and every code must be within one of the GPU's,
  every scale within one bf16 ulp of absmax / 7, with almost all equal (the
  GPU rotates in fp32, the oracle in fp64, so the bf16 rounding of a rotated
  value can differ by one ulp); every position of every sequence for phi3,
  gqa and mixed, every eighth sequence of the long-context batch; spare
  blocks keep their sentinel bytes;
* end to end, sampled: the oracle's own write of sampled sequences, then its
  attention, against the GPU output (codes may differ by one between the two
  writes), correlation >= 0.9999 over the sampled rows together.
"""

import math
import os
import shutil
import time

import numpy as np
import pytest
import torch

from int4_token_head_gb300 import synthetic
from int4_token_head_gb300.paged import PagedKV
from tests import oracle_pool as P
from tests.helpers import assert_close_attention, check_sampled_end_to_end, corr

pytestmark = pytest.mark.gpu

WORKLOADS = ["phi3", "gqa", "gqa_window1000", "mixed", "long"]


def _bits(t):
    """bf16 tensor -> uint16 numpy array of its bit patterns (on the host)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def _dump_caches(pk, directory, chunk_blocks=16384):
    """Copy the four cache tensors into .npy files, a chunk of blocks at a time."""
    for name in ("k_cache", "v_cache", "k_scale", "v_scale"):
        t = getattr(pk, name)
        dtype = np.uint8 if t.dtype == torch.uint8 else np.float32
        mm = np.lib.format.open_memmap(os.path.join(directory, f"{name}.npy"), mode="w+", dtype=dtype,
                                       shape=tuple(t.shape))
        for b0 in range(0, t.shape[0], chunk_blocks):
            mm[b0:b0 + chunk_blocks] = t[b0:b0 + chunk_blocks].cpu().numpy()
        mm.flush()
        del mm


def _run_step(name):
    if name == "gqa_window1000":
        w = synthetic.make_workload("gqa")
        w.sliding_window = 1000
    else:
        w = synthetic.make_workload(name)
    pk = PagedKV(w)
    pk.populate_history()
    q, k, v, slots = pk.step_inputs()
    out = torch.full((w.num_q_tokens, w.num_q_heads, w.head_size), float("nan"), dtype=torch.bfloat16,
                     device="cuda")
    pk.step(q, k, v, slots, out)
    torch.cuda.synchronize()
    assert pk.status.item() == 0
    return w, pk, q, out


def _write_sequences(w):
    """Sequences whose every position is checked code by code."""
    if w.name == "long":
        return list(range(0, w.num_seqs, 8))
    return list(range(w.num_seqs))


@pytest.mark.parametrize("name", WORKLOADS)
def test_full_size_whole_output(name):
    t0 = time.time()
    w, pk, q, out = _run_step(name)
    got = out.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    q_bits = _bits(q)
    bt = w.block_table.numpy()
    signs = w.signs.numpy().astype(np.float64)
    scale = 1.0 / math.sqrt(w.head_size)
    G = w.group
    nbytes = sum(t.numel() * t.element_size() for t in (pk.k_cache, pk.v_cache, pk.k_scale, pk.v_scale))
    directory = P.scratch_dir(nbytes)
    try:
        _dump_caches(pk, directory)
        t_dump = time.time()
        qsl = w.query_start_loc.numpy()
        with P.oracle_pool() as pool:
            # ---- attention alone over the GPU-written cache: every (sequence, kv head) ----
            units, where = [], []
            for s, (ql, L) in enumerate(w.seqs):
                if ql == 0:
                    continue
                q0 = int(qsl[s])
                for h in range(w.num_kv_heads):
                    units.append((directory, q_bits[q0:q0 + ql, h * G:(h + 1) * G], bt[s], L, ql, h, G,
                                  w.num_kv_heads, w.block_size, scale, w.causal, signs, w.sliding_window))
                    where.append((q0, ql, h))
            ref = np.full_like(got, np.nan)
            for (q0, ql, h), r in zip(where, pool.imap(P.attention_unit, units, chunksize=4)):
                ref[q0:q0 + ql, h * G:(h + 1) * G] = r
            t_attn = time.time()
            assert np.isfinite(ref).all()
            max_err, c = assert_close_attention(got, ref, what=f"{name} whole output")
            rows_got = got.reshape(-1, w.head_size)
            rows_ref = ref.reshape(-1, w.head_size)
            row_corr = min(corr(a, b) for a, b in zip(rows_got, rows_ref))
            # every (token, q head) row on its own, too (measured minimum 0.999996)
            assert row_corr >= 0.9999, f"{name}: a row correlates {row_corr:.6f} with the oracle"

            # ---- the write, code by code, from the same K/V ----
            summary = None
            if name != "gqa_window1000":  # the same cache as gqa
                summary = np.zeros((2, 6), dtype=np.float64)
                seqs = _write_sequences(w)
                batch = []

                def flush():
                    for res in pool.map(P.write_unit, batch):
                        for i, r in enumerate(res):
                            summary[i, 0] = max(summary[i, 0], r[0])
                            summary[i, 1:3] += r[1:3]
                            summary[i, 3] = max(summary[i, 3], r[3])
                            summary[i, 4:6] += r[4:6]
                    batch.clear()

                for s in seqs:
                    _, L = w.seqs[s]
                    k, v = w.seq_kv(s, "cuda")
                    kb, vb = _bits(k), _bits(v)
                    for p0 in range(0, L, 4096):
                        p1 = min(L, p0 + 4096)
                        rows = bt[s][p0 // 16:(p1 + 15) // 16]
                        batch.append((directory, kb[p0:p1], vb[p0:p1], rows, w.block_size, signs))
                        if len(batch) >= 4 * P.host_processes():
                            flush()
                flush()
        t_write = time.time()
        if summary is not None:
            for i, which in enumerate(("K", "V")):
                code_max, code_diff, n_codes, scale_rel, scale_diff, n_scales = summary[i]
                assert code_max <= 1, f"{name} {which}: a code differs by {code_max}"
                assert code_diff / n_codes < 1e-3, f"{name} {which}: {code_diff} of {n_codes} codes differ"
                assert scale_rel <= 2.0 ** -7, f"{name} {which}: scale off by {scale_rel:.3g} (relative)"
                assert scale_diff / n_scales < 1e-2, f"{name} {which}: {scale_diff} of {n_scales} scales differ"
            # blocks no sequence owns keep their sentinel bytes
            used = set(int(b) for b in bt.ravel() if b >= 0)
            spare = [b for b in range(w.num_blocks) if b not in used]
            if spare:
                sp = torch.tensor(spare, dtype=torch.int64, device="cuda")
                assert bool((pk.k_cache[sp] == synthetic.SENTINEL_CODE_BYTE).all())
                assert bool((pk.v_cache[sp] == synthetic.SENTINEL_CODE_BYTE).all())
                bits = pk.k_scale[sp].view(torch.int32)
                assert bool((bits == synthetic.SENTINEL_SCALE_BITS).all())
    finally:
        shutil.rmtree(directory, ignore_errors=True)

    # ---- end to end on sampled sequences (the oracle's own write) ----
    if w.name == "mixed":
        pre = [s for s, (ql, _) in enumerate(w.seqs) if ql > 1][:2]
        dec = [s for s, (ql, _) in enumerate(w.seqs) if ql == 1][:2]
        sample = pre + dec
    else:
        sample = [0, w.num_seqs // 2, w.num_seqs - 1]
    e2e_err, e2e_corr = check_sampled_end_to_end(w, q, out, seqs=sample, heads=[0, w.num_q_heads - 1])
    print(f"{name}: whole output max abs err {max_err:.4g}, corr {c:.7f}, min row corr {row_corr:.6f}; "
          f"write {summary.tolist() if summary is not None else 'as gqa'}; end to end sampled max err "
          f"{e2e_err:.4g} corr {e2e_corr:.7f}; times: step+dump {t_dump - t0:.1f}s, attention oracle "
          f"{t_attn - t_dump:.1f}s, write oracle {t_write - t_attn:.1f}s on {P.host_processes()} processes")
    del pk
    torch.cuda.empty_cache()
