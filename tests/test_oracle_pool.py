"""The process-pool workers of the full-size parity tests give the oracle's
own results: attention per (sequence, kv head) unit over a dumped cache
equals the oracle's whole-batch attention, and the write comparison finds no
difference on the oracle's own cache and exactly the differences planted in
a copy of it.  CPU only (a small mixed workload written by the oracle)."""

import math
import os
import shutil

import numpy as np

from oracle import kvint4_oracle as O
from int4_token_head_gb300 import synthetic
from tests import oracle_pool as P
from tests.helpers import oracle_write_history_and_step


def _dump(caches, directory):
    for name, arr in zip(("k_cache", "v_cache", "k_scale", "v_scale"), caches):
        np.save(os.path.join(directory, f"{name}.npy"), arr)


def _bits(t):
    import torch
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def test_pool_units_reproduce_the_oracle():
    w = synthetic.custom_workload(8, 2, 96, [(1, 70), (20, 40), (1, 17)], seed=31, sliding_window=0)
    caches = oracle_write_history_and_step(w)
    q = w.queries("cpu")
    scale = 1.0 / math.sqrt(w.head_size)
    ref = O.attention(q.float().numpy(), *caches, w.block_table.numpy(), w.seq_lens.numpy(),
                      w.query_start_loc.numpy(), w.num_kv_heads, w.block_size, scale, True, w.signs.numpy())
    directory = P.scratch_dir(1 << 20)
    try:
        _dump(caches, directory)
        G, qsl, bt = w.group, w.query_start_loc.numpy(), w.block_table.numpy()
        signs = w.signs.numpy().astype(np.float64)
        qb = _bits(q)
        units, where = [], []
        for s, (ql, L) in enumerate(w.seqs):
            q0 = int(qsl[s])
            for h in range(w.num_kv_heads):
                units.append((directory, qb[q0:q0 + ql, h * G:(h + 1) * G], bt[s], L, ql, h, G, w.num_kv_heads,
                              16, scale, True, signs, 0))
                where.append((q0, ql, h))
        with P.oracle_pool(2) as pool:
            got = np.full_like(ref, np.nan)
            for (q0, ql, h), r in zip(where, pool.map(P.attention_unit, units)):
                got[q0:q0 + ql, h * G:(h + 1) * G] = r
            assert np.array_equal(got, ref)

            # the write comparison: no difference on the oracle's own cache ...
            args = []
            for s, (ql, L) in enumerate(w.seqs):
                k, v = w.seq_kv(s, "cpu")
                args.append((directory, _bits(k), _bits(v), bt[s], 16, signs))
            for res in pool.map(P.write_unit, args):
                for code_max, code_diff, n, rel, sdiff, ns in res:
                    assert code_max == 0 and code_diff == 0 and rel == 0 and sdiff == 0 and n > 0 and ns > 0
            # ... and exactly the planted ones in a modified copy
            kc = caches[0].copy()
            blk0 = bt[0][0]
            kc[blk0, 3, 1, 5] ^= 0x01          # one code of sequence 0, position 3, kv head 1: +-1
            vs = caches[3].copy()
            vs[blk0, 4, 0] *= np.float32(1 + 2.0 ** -8)
            _dump((kc, caches[1], caches[2], vs), directory)
            res = pool.map(P.write_unit, args[:1])[0]
            assert res[0][0] == 1 and res[0][1] == 1
            assert res[1][4] == 1 and 0 < res[1][3] <= 2.0 ** -7
    finally:
        shutil.rmtree(directory, ignore_errors=True)
