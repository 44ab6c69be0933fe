"""Process-pool workers that run the fp64 oracle over a GPU-written paged
cache, for the full-size parity tests.

Test infrastructure: this module imports numpy and the oracle only (never
torch or the CUDA library), so spawned workers start quickly and never touch
a GPU.  The caches are handed over as .npy files that every worker maps
read-only; K/V values travel as bf16 bit patterns (uint16).
"""

from __future__ import annotations

import contextlib
import multiprocessing as mp
import os
import shutil
import tempfile

import numpy as np

from oracle import kvint4_oracle as O

_CACHES = {}


def _caches(cache_dir):
    """(k_cache, v_cache, k_scale, v_scale) of a dumped cache, memory-mapped once per worker."""
    c = _CACHES.get(cache_dir)
    if c is None:
        c = tuple(np.load(os.path.join(cache_dir, f"{n}.npy"), mmap_mode="r")
                  for n in ("k_cache", "v_cache", "k_scale", "v_scale"))
        _CACHES.clear()
        _CACHES[cache_dir] = c
    return c


def bf16_bits_to_f64(u16):
    """bf16 bit patterns (uint16) -> float64 values (exact)."""
    u = np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def attention_unit(args):
    """Oracle output rows [q_len, G, d] of one (sequence, kv head) unit over the dumped cache."""
    (cache_dir, q_rows_bits, bt_row, L, ql, kv_head, group, hkv, block_size, scale, causal, signs, window) = args
    kc, vc, ks, vs = _caches(cache_dir)
    q = bf16_bits_to_f64(q_rows_bits)  # [ql, G, d]
    d = q.shape[-1]
    codes_k, sk = O.gather_sequence(kc, ks, bt_row, L, kv_head, block_size)
    codes_v, sv = O.gather_sequence(vc, vs, bt_row, L, kv_head, block_size)
    k_hat = O.dequantize_original(codes_k, sk, signs)
    v_hat = O.dequantize_original(codes_v, sv, signs)
    out = np.empty((ql, group, d))
    for j in range(group):
        out[:, j, :] = O.attention_head(q[:, j, :], k_hat, v_hat, L - ql, scale, causal, window)
    return out


def write_unit(args):
    """Compare the dumped cache rows of positions [0, L) of one sequence with
    the oracle's quantisation of the same K/V.  Returns per-tensor summaries:
    (max |code diff|, number of differing codes, number of codes, max relative
    scale difference, number of differing scales, number of scales)."""
    cache_dir, k_bits, v_bits, bt_row, block_size, signs = args
    kc, vc, ks, vs = _caches(cache_dir)
    L = k_bits.shape[0]
    pos = np.arange(L)
    blk = np.asarray(bt_row, dtype=np.int64)[pos // block_size]
    off = pos % block_size
    res = []
    for bits, cache, scale in ((k_bits, kc, ks), (v_bits, vc, vs)):
        x = bf16_bits_to_f64(bits)  # [L, Hkv, d]
        codes, s = O.quantize(O.rotate_for_cache(x, signs))
        got_codes = O.unpack_codes(np.asarray(cache[blk, off])).astype(np.int32)
        got_s = np.asarray(scale[blk, off]).astype(np.float64)
        diff = np.abs(got_codes - codes.astype(np.int32))
        ref_s = s.astype(np.float64)
        with np.errstate(divide="ignore", invalid="ignore"):
            rel = np.where(ref_s > 0, np.abs(got_s - ref_s) / ref_s, np.abs(got_s - ref_s))
        res.append((int(diff.max()) if diff.size else 0, int((diff != 0).sum()), int(diff.size),
                    float(np.nanmax(rel)) if rel.size else 0.0, int((got_s != ref_s).sum()), int(ref_s.size)))
    return res


def scratch_dir(nbytes):
    """A fresh directory with room for nbytes: /dev/shm when it has room, else the temp dir."""
    for base in ("/dev/shm", tempfile.gettempdir()):
        try:
            if os.path.isdir(base) and shutil.disk_usage(base).free > 1.2 * nbytes + (1 << 30):
                return tempfile.mkdtemp(prefix="kvint4_parity_", dir=base)
        except OSError:
            continue
    raise RuntimeError(f"no scratch directory with {nbytes / 1e9:.1f} GB free for the cache dump")


def host_processes():
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:
        n = os.cpu_count() or 1
    return max(1, min(n, 64))


@contextlib.contextmanager
def oracle_pool(processes=None):
    """A spawn pool (safe after CUDA initialisation) whose workers each use one
    BLAS thread."""
    keys = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
    saved = {k: os.environ.get(k) for k in keys}
    for k in keys:
        os.environ[k] = "1"
    try:
        pool = mp.get_context("spawn").Pool(processes or host_processes())
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    try:
        yield pool
    finally:
        pool.terminate()
        pool.join()
