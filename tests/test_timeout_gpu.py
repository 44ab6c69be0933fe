"""The bounded barrier wait of the pipelined kernels, exercised on a GPU
without a fault or a hang: a warp waits on an mbarrier that nothing arrives
at (kv_int4_selftest_wait), gives up after its attempts, reports
KV_INT4_DEV_TIMEOUT, and the context stays usable afterwards."""

import time

import pytest
import torch

from int4_token_head_gb300 import _lib, synthetic
from int4_token_head_gb300.paged import PagedKV
from tests.helpers import assert_close_attention, oracle_attention, oracle_write_history_and_step

pytestmark = pytest.mark.gpu
KERNEL_LIMIT = 1 << 18  # attempts of the kernels' bounded waits


def _wait(iterations):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cycles = torch.zeros(1, dtype=torch.int64, device="cuda")
    t0 = time.perf_counter()
    _lib.selftest_wait(iterations, status, cycles)
    torch.cuda.synchronize()
    return int(status.item()), int(cycles.item()), time.perf_counter() - t0


def test_bounded_wait_reports_time_out_and_the_context_stays_usable():
    status, cycles, _ = _wait(4096)
    assert status == _lib.DEV_TIMEOUT
    assert cycles > 0
    per_attempt = cycles / 4096
    # the kernels' own limit ends within seconds at this rate (SM clocks >= 1 GHz)
    assert per_attempt * KERNEL_LIMIT / 1e9 < 10.0, per_attempt
    # the full limit itself: the wait ends, reports, and the stream moves on
    status, cycles, wall = _wait(KERNEL_LIMIT)
    assert status == _lib.DEV_TIMEOUT and wall < 10.0
    print(f"bounded wait: {per_attempt:.0f} SM cycles per attempt; the kernels' limit "
          f"({KERNEL_LIMIT} attempts) held the warp {cycles} cycles, {wall * 1e3:.0f} ms wall")
    # a zero budget gives up at once (and says so)
    status, _, _ = _wait(0)
    assert status == _lib.DEV_TIMEOUT
    # the context is intact: a prefill (pipelined kernel with bounded waits) matches the oracle
    w = synthetic.custom_workload(16, 4, 128, [(70, 100), (1, 40)], seed=61)
    caches = oracle_write_history_and_step(w)
    pk = PagedKV(w)
    for dst, src in zip((pk.k_cache, pk.v_cache, pk.k_scale, pk.v_scale), caches):
        dst.copy_(torch.from_numpy(src))
    q = w.queries("cpu")
    out = torch.full((w.num_q_tokens, w.num_q_heads, w.head_size), float("nan"), dtype=torch.bfloat16, device="cuda")
    pk.attend(q.cuda(), out)
    torch.cuda.synchronize()
    assert pk.status.item() == 0
    assert_close_attention(out.float().cpu().numpy(), oracle_attention(w, q, caches), what="after time-out")
