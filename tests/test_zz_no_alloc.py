"""kv_int4_attention_noalloc: attention for callers that cannot allocate
device memory (a framework or plugin host that owns every allocation, or a
pipeline that may not call cudaMalloc once running).  It uses the library's
static device scratch instead of a caller workspace; its results must match
the regular entry point's, call after call, since every call reuses the same
scratch with the previous call's contents still in it.

This file is collected last on purpose.
"""

import numpy as np
import pytest
import torch

from int4_token_head_gb300 import _lib, synthetic
from int4_token_head_gb300.paged import PagedKV
from tests.helpers import assert_close_attention


def _prepared(w):
    pk = PagedKV(w)
    pk.populate_history(gen_device="cpu")
    q, k, v, slots = pk.step_inputs(gen_device="cpu")
    pk.write(k, v, slots)
    return pk, q


def _noalloc(pk, q, out):
    w = pk.w
    _lib.attention_noalloc(q, pk.k_cache, pk.v_cache, pk.k_scale, pk.v_scale, pk.block_table, pk.seq_lens,
                           pk.query_start_loc, w.max_query_len, w.max_seq_len, pk.softmax_scale, w.causal,
                           pk.signs, out, dev_status=pk.status)


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    cases = [
        synthetic.custom_workload(16, 4, 192, [(1, 300), (60, 60), (1, 45), (25, 200), (1, 1)], seed=21),
        synthetic.custom_workload(32, 8, 128, [(1, 700), (1, 33), (2, 90), (1, 1500)], seed=22),
    ]
    prepared = [_prepared(w) for w in cases]
    refs = []
    for pk, q in prepared:
        ref = torch.empty((q.shape[0], pk.w.num_q_heads, pk.w.head_size), dtype=torch.bfloat16, device="cuda")
        pk.attend(q, ref)  # the existing entry point, with a caller workspace
        refs.append(ref)
    torch.cuda.synchronize()
    # two calls in a row on each shape, alternating shapes so that each call
    # starts from scratch contents another shape left behind
    for rnd in range(2):
        for (pk, q), ref in zip(prepared, refs):
            out = torch.full_like(ref, float("nan"))
            _noalloc(pk, q, out)
            torch.cuda.synchronize()
            assert pk.status.item() == 0
            got = out.float().cpu().numpy()
            want = ref.float().cpu().numpy()
            assert_close_attention(got, want, what=f"noalloc round {rnd} {pk.w.head_size}")
            assert np.array_equal(got, want)  # same kernels, same schedule


def test_noalloc_rejects_sizes_beyond_the_scratch():
    lib = _lib.load()
    need = lib.kv_int4_attention_workspace_size(100000, 100000, 64, 8, 256)
    assert need > _lib.NOALLOC_SCRATCH_BYTES
    fake = __import__("ctypes").c_void_p(0x10000)
    rc = lib.kv_int4_attention_noalloc(fake, 64 * 256, fake, fake, fake, fake, fake, 8, fake, fake, 100000, 100000,
                                       1, 128, 64, 8, 256, 16, 16, 0.1, 1, 0, fake, fake, 64 * 256, None, None)
    assert rc == _lib.ERR_SCRATCH_LIMIT
    assert "no-allocation scratch" in _lib.status_string(rc)
