"""Host threads may call the library concurrently: launch settings (shared
memory limits, occupancies) are computed once per device context under a
lock.  A fresh process (so that every setting starts uncomputed) runs the
write, the attention (decode, tensor-core prefill, mma.sync prefill) and the
standalone rotation from eight threads at once, each on its own stream with
its own buffers; every result must equal, bit for bit, the result of the same
calls made afterwards from one thread."""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import threading
import torch
from int4_token_head_gb300 import _lib, synthetic
from int4_token_head_gb300.paged import PagedKV

torch.cuda.set_device(0)
_lib.load()
shapes = [(16, 4, 192, [(1, 300), (60, 60), (1, 45)]), (32, 8, 128, [(1, 700), (1, 33)]),
          (4, 2, 256, [(30, 64), (1, 100)]), (8, 8, 96, [(1, 200), (20, 90)])]
jobs = []
for i in range(8):
    hq, hkv, d, seqs = shapes[i % len(shapes)]
    w = synthetic.custom_workload(hq, hkv, d, seqs, seed=70 + i)
    pk = PagedKV(w)
    hist = w.history_kv("cuda")
    q, k, v, slots = pk.step_inputs()
    x = torch.randn((999, d), device="cuda").to(torch.bfloat16)
    jobs.append(dict(w=w, pk=pk, hist=hist, hslots=w.history_slot_mapping().cuda(), step=(q, k, v, slots), x=x,
                     stream=torch.cuda.Stream()))
torch.cuda.synchronize()

def run(j, out, y):
    pk = j["pk"]
    q, k, v, slots = j["step"]
    with torch.cuda.stream(j["stream"]):
        pk.write(j["hist"][0], j["hist"][1], j["hslots"], stream=j["stream"])
        pk.step(q, k, v, slots, out, stream=j["stream"])
        _lib.rht(j["x"], pk.signs, out=y, stream=j["stream"])

outs, ys = [], []
for j in jobs:
    w = j["w"]
    outs.append(torch.empty((w.num_q_tokens, w.num_q_heads, w.head_size), dtype=torch.bfloat16, device="cuda"))
    ys.append(torch.empty_like(j["x"]))
gate = threading.Barrier(len(jobs))
errors = []

def worker(i):
    try:
        gate.wait()
        run(jobs[i], outs[i], ys[i])
    except Exception as e:
        errors.append(repr(e))

threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(jobs))]
for t in threads:
    t.start()
for t in threads:
    t.join()
torch.cuda.synchronize()
assert not errors, errors
for i, j in enumerate(jobs):
    assert j["pk"].status.item() == 0, i
    caches = [t.clone() for t in (j["pk"].k_cache, j["pk"].v_cache, j["pk"].k_scale, j["pk"].v_scale)]
    out2, y2 = torch.empty_like(outs[i]), torch.empty_like(ys[i])
    run(j, out2, y2)
    torch.cuda.synchronize()
    assert torch.equal(out2, outs[i]), f"attention of job {i}"
    assert torch.equal(y2, ys[i]), f"rotation of job {i}"
    for a, b in zip(caches, (j["pk"].k_cache, j["pk"].v_cache, j["pk"].k_scale, j["pk"].v_scale)):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), f"cache of job {i}"
print("threads ok")
"""


def test_concurrent_first_calls_from_host_threads():
    r = subprocess.run([sys.executable, "-c", SCRIPT], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "threads ok" in r.stdout
