"""ctypes binding of libkvint4.so: argument marshalling only.

Every function takes torch tensors, checks dtypes/shapes/layouts, and passes
raw device pointers and sizes to the C ABI declared in include/kvint4.h.  All
computation happens in the library's CUDA kernels; if the library cannot be
built or loaded, these functions raise instead of computing anything else.
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import build as _build

_lock = threading.Lock()
_lib = None

c_int, c_int64, c_void_p, c_size_t, c_float = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_float

_SIGNATURES = {
    "kv_int4_write": (c_int, [c_void_p, c_int64, c_void_p, c_int64, c_void_p, c_int, c_void_p, c_void_p,
                              c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_void_p, c_void_p, c_void_p]),
    "kv_int4_write_prerotated": (c_int, [c_void_p, c_int64, c_void_p, c_int64, c_void_p, c_int, c_void_p,
                                         c_void_p, c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_void_p,
                                         c_void_p]),
    "kv_int8_write": (c_int, [c_void_p, c_int64, c_void_p, c_int64, c_void_p, c_int, c_void_p, c_void_p,
                              c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_void_p, c_void_p]),
    "kv_int4_attention_workspace_size": (c_size_t, [c_int, c_int, c_int, c_int, c_int]),
    "kv_int4_attention": (c_int, [c_void_p, c_int64, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int,
                                  c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_int,
                                  c_int, c_float, c_int, c_int, c_void_p, c_void_p, c_int64, c_void_p, c_size_t,
                                  c_void_p, c_void_p]),
    "kv_int4_attention_noalloc": (c_int, [c_void_p, c_int64, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                          c_int, c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int, c_int,
                                          c_int, c_int, c_int, c_float, c_int, c_int, c_void_p, c_void_p, c_int64,
                                          c_void_p, c_void_p]),
    "kv_int4_rht": (c_int, [c_void_p, c_int64, c_void_p, c_int64, c_int, c_int64, c_int, c_void_p, c_int, c_void_p]),
    "kv_int8_attention": (c_int, [c_void_p, c_int64, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int,
                                  c_void_p, c_void_p, c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_int,
                                  c_int, c_float, c_int, c_int, c_void_p, c_int64, c_void_p, c_size_t,
                                  c_void_p, c_void_p]),
    "kv_int4_inslot_slot_bytes": (c_int, [c_int, c_int]),
    "kv_int4_write_inslot": (c_int, [c_void_p, c_int64, c_void_p, c_int64, c_void_p, c_int, c_void_p, c_int, c_int,
                                     c_int, c_int, c_void_p, c_void_p, c_void_p]),
    "kv_int8_write_inslot": (c_int, [c_void_p, c_int64, c_void_p, c_int64, c_void_p, c_int, c_void_p, c_int, c_int,
                                     c_int, c_int, c_void_p, c_void_p]),
    "kv_int4_attention_inslot": (c_int, [c_void_p, c_int64, c_void_p, c_void_p, c_int, c_void_p, c_void_p, c_int,
                                         c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_float, c_int,
                                         c_int, c_void_p, c_void_p, c_int64, c_void_p, c_size_t, c_void_p,
                                         c_void_p]),
    "kv_int8_attention_inslot": (c_int, [c_void_p, c_int64, c_void_p, c_void_p, c_int, c_void_p, c_void_p, c_int,
                                         c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_int, c_float, c_int,
                                         c_int, c_void_p, c_int64, c_void_p, c_size_t, c_void_p, c_void_p]),
    "kv_int4_status_string": (ctypes.c_char_p, [c_int]),
    "kv_int4_timing_enable": (c_int, [c_int]),
    "kv_int4_timing_collect": (c_int, [c_void_p, c_void_p, c_void_p]),
    "kv_int4_selftest_wait": (c_int, [c_int, c_void_p, c_void_p, c_void_p]),
    "kv_int4_version": (c_int, []),
}

OK = 0
ERR_SCRATCH_LIMIT = 9
NOALLOC_SCRATCH_BYTES = 64 << 20
DEV_BAD_SLOT, DEV_BAD_BLOCK, DEV_BAD_SEQ, DEV_BAD_SIGNS, DEV_TIMEOUT = 1, 2, 4, 8, 16


class KvInt4Error(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} (status {code})")


def load(path: Optional[str] = None):
    """Load (building first if needed) libkvint4.so and declare its signatures."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        # KVINT4_LIBRARY selects a specific build of the library (for example a
        # locally modified one); otherwise the in-tree library is built if stale.
        p = path or os.environ.get("KVINT4_LIBRARY") or _build.build()
        lib = ctypes.CDLL(p)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path is None:
            _lib = lib
        return lib


def library_path() -> str:
    return _build.LIB_PATH


def status_string(code: int) -> str:
    return load().kv_int4_status_string(int(code)).decode()


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _check(cond, msg):
    if not cond:
        raise ValueError(msg)


def _token_major(x: torch.Tensor, name: str, heads: int, d: int):
    _check(x.dim() == 3 and x.shape[1] == heads and x.shape[2] == d,
           f"{name} must be [tokens, {heads}, {d}], got {tuple(x.shape)}")
    _check(x.dtype == torch.bfloat16, f"{name} must be bfloat16")
    _check(x.stride(2) == 1 and (x.shape[1] <= 1 or x.stride(1) == d),
           f"{name} must have contiguous heads and head dims")
    return x.stride(0) if x.shape[0] > 0 else heads * d


def _cache_dims(k_cache, v_cache, k_scale, v_scale):
    _check(k_cache.dtype == torch.uint8 and v_cache.dtype == torch.uint8, "caches must be uint8")
    _check(k_cache.dim() == 4 and k_cache.shape == v_cache.shape, "caches must be [blocks, block_size, heads, d/2]")
    _check(k_cache.is_contiguous() and v_cache.is_contiguous(), "caches must be contiguous")
    nb, bs, hkv, half = k_cache.shape
    for s in (k_scale, v_scale):
        _check(s.dtype == torch.float32 and tuple(s.shape) == (nb, bs, hkv) and s.is_contiguous(),
               "scale caches must be contiguous float32 [blocks, block_size, heads]")
    return nb, bs, hkv, 2 * half


def _raise(code, where):
    if code != OK:
        raise KvInt4Error(code, where)


def write(k, v, slot_mapping, k_cache, v_cache, k_scale, v_scale, signs,
          dev_status: Optional[torch.Tensor] = None, stream=None, prerotated: bool = False):
    """reshape_and_cache_int4 through kv_int4_write (or kv_int4_write_prerotated)."""
    nb, bs, hkv, d = _cache_dims(k_cache, v_cache, k_scale, v_scale)
    ks = _token_major(k, "k", hkv, d)
    vs = _token_major(v, "v", hkv, d)
    _check(k.shape[0] == v.shape[0] == slot_mapping.shape[0], "k, v and slot_mapping disagree on tokens")
    _check(slot_mapping.dtype == torch.int64 and slot_mapping.is_contiguous(), "slot_mapping must be contiguous int64")
    lib = load()
    if prerotated:
        code = lib.kv_int4_write_prerotated(_ptr(k), ks, _ptr(v), vs, _ptr(slot_mapping), int(k.shape[0]),
                                            _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                            nb, bs, hkv, d, _ptr(dev_status), _stream(stream))
        _raise(code, "kv_int4_write_prerotated")
    else:
        _check(signs.dtype == torch.int8 and signs.numel() == d and signs.is_contiguous(), "signs must be int8 [d]")
        code = lib.kv_int4_write(_ptr(k), ks, _ptr(v), vs, _ptr(slot_mapping), int(k.shape[0]),
                                 _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                 nb, bs, hkv, d, _ptr(signs), _ptr(dev_status), _stream(stream))
        _raise(code, "kv_int4_write")


def rht(x, signs, inverse: bool = False, out: Optional[torch.Tensor] = None,
        out_dtype: torch.dtype = torch.bfloat16, stream=None) -> torch.Tensor:
    """The block-diagonal randomized Hadamard rotation through kv_int4_rht.

    x: bf16 [..., d] with a contiguous last dimension (rows may be strided);
    forward y = (I_n (x) H_b) D x, inverse y = D (I_n (x) H_b) x / b.  The
    result (bf16 or float32, shape of x) is written to `out` if given."""
    _check(x.dtype == torch.bfloat16, "x must be bfloat16")
    _check(x.dim() >= 1 and x.stride(-1) == 1, "x must have a contiguous last dimension")
    d = x.shape[-1]
    rows = x.numel() // d if d else 0
    x2 = x.reshape(rows, d) if x.dim() != 2 else x
    _check(signs.dtype == torch.int8 and signs.numel() == d and signs.is_contiguous(), "signs must be int8 [d]")
    if out is None:
        out = torch.empty(x.shape, dtype=out_dtype, device=x.device)
    _check(out.dtype in (torch.bfloat16, torch.float32), "out must be bfloat16 or float32")
    _check(tuple(out.shape) == tuple(x.shape) and out.stride(-1) == 1, "out must match x's shape, last dim contiguous")
    o2 = out.reshape(rows, d) if out.dim() != 2 else out
    _check(o2.data_ptr() == out.data_ptr(), "out must be viewable as rows")
    xs = x2.stride(0) if rows > 1 else d
    ys = o2.stride(0) if rows > 1 else d
    code = load().kv_int4_rht(_ptr(x2), xs, _ptr(o2), ys, int(out.dtype == torch.float32), rows, d, _ptr(signs),
                              int(bool(inverse)), _stream(stream))
    _raise(code, "kv_int4_rht")
    return out


def _cache_dims_int8(k_cache, v_cache, k_scale, v_scale):
    _check(k_cache.dtype == torch.int8 and v_cache.dtype == torch.int8, "int8 caches must be int8")
    _check(k_cache.dim() == 4 and k_cache.shape == v_cache.shape, "caches must be [blocks, block_size, heads, d]")
    _check(k_cache.is_contiguous() and v_cache.is_contiguous(), "caches must be contiguous")
    nb, bs, hkv, d = k_cache.shape
    for s in (k_scale, v_scale):
        _check(s.dtype == torch.float32 and tuple(s.shape) == (nb, bs, hkv) and s.is_contiguous(),
               "scale caches must be contiguous float32 [blocks, block_size, heads]")
    return nb, bs, hkv, d


def write_int8(k, v, slot_mapping, k_cache, v_cache, k_scale, v_scale,
               dev_status: Optional[torch.Tensor] = None, stream=None):
    """The int8_per_token_head write (no rotation) through kv_int8_write."""
    nb, bs, hkv, d = _cache_dims_int8(k_cache, v_cache, k_scale, v_scale)
    ks = _token_major(k, "k", hkv, d)
    vs = _token_major(v, "v", hkv, d)
    _check(k.shape[0] == v.shape[0] == slot_mapping.shape[0], "k, v and slot_mapping disagree on tokens")
    _check(slot_mapping.dtype == torch.int64 and slot_mapping.is_contiguous(), "slot_mapping must be contiguous int64")
    code = load().kv_int8_write(_ptr(k), ks, _ptr(v), vs, _ptr(slot_mapping), int(k.shape[0]), _ptr(k_cache),
                                _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), nb, bs, hkv, d, _ptr(dev_status),
                                _stream(stream))
    _raise(code, "kv_int8_write")


TIMED_KINDS = ("write", "prep", "prefill", "decode", "reduce")


def timing_enable(enable: bool = True):
    """Record CUDA events around every kernel the library launches from this thread."""
    load().kv_int4_timing_enable(int(bool(enable)))


def timing_collect():
    """{kind: (total_ms, launches, dropped)} since the last collect (waits for the events)."""
    n = len(TIMED_KINDS)
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_int * n)()
    drop = (ctypes.c_int * n)()
    _raise(load().kv_int4_timing_collect(ms, cnt, drop), "kv_int4_timing_collect")
    return {k: (ms[i], cnt[i], drop[i]) for i, k in enumerate(TIMED_KINDS)}


def selftest_wait(iterations: int, dev_status: torch.Tensor, dev_cycles: Optional[torch.Tensor] = None, stream=None):
    """One warp waits on an mbarrier nothing arrives at, gives up after `iterations`
    attempts and ORs DEV_TIMEOUT into dev_status (int32 [1]); dev_cycles (int64 [1])
    receives the SM cycles it waited."""
    _check(dev_status.dtype == torch.int32 and dev_status.is_cuda, "dev_status: int32 CUDA tensor")
    _check(dev_cycles is None or (dev_cycles.dtype == torch.int64 and dev_cycles.is_cuda), "dev_cycles: int64 CUDA tensor")
    _raise(load().kv_int4_selftest_wait(int(iterations), _ptr(dev_status), _ptr(dev_cycles), _stream(stream)),
           "kv_int4_selftest_wait")


def attention_workspace_size(num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_size) -> int:
    return int(load().kv_int4_attention_workspace_size(num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_size))


def attention(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, query_start_loc,
              max_query_len, max_seq_len, softmax_scale, causal, signs, out, workspace,
              dev_status: Optional[torch.Tensor] = None, stream=None, sliding_window: int = 0):
    """unified_attention_int4 through kv_int4_attention; writes ``out`` in place.
    ``sliding_window`` W > 0 hides keys at positions <= p - W from the query at p."""
    nb, bs, hkv, d = _cache_dims(k_cache, v_cache, k_scale, v_scale)
    _check(q.dim() == 3 and q.shape[2] == d, "q must be [tokens, q_heads, d]")
    hq = q.shape[1]
    qs = _token_major(q, "q", hq, d)
    os_ = _token_major(out, "out", hq, d)
    _check(out.shape[0] == q.shape[0], "out must match q")
    _check(block_table.dtype == torch.int32 and block_table.dim() == 2 and block_table.is_contiguous(),
           "block_table must be contiguous int32 [seqs, max_blocks]")
    _check(seq_lens.dtype == torch.int32 and query_start_loc.dtype == torch.int32, "seq_lens/query_start_loc int32")
    num_seqs = seq_lens.shape[0]
    _check(query_start_loc.shape[0] == num_seqs + 1 and block_table.shape[0] == num_seqs, "metadata shapes")
    _check(signs.dtype == torch.int8 and signs.numel() == d, "signs must be int8 [d]")
    _check(workspace.dtype == torch.uint8 and workspace.is_contiguous(), "workspace must be contiguous uint8")
    lib = load()
    code = lib.kv_int4_attention(_ptr(q), qs, _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                 _ptr(block_table), int(block_table.shape[1]), _ptr(seq_lens),
                                 _ptr(query_start_loc), int(num_seqs), int(q.shape[0]), int(max_query_len),
                                 int(max_seq_len), int(hq), int(hkv), int(d), int(bs), int(nb),
                                 float(softmax_scale), int(bool(causal)), int(sliding_window), _ptr(signs),
                                 _ptr(out), os_, _ptr(workspace), int(workspace.numel()), _ptr(dev_status),
                                 _stream(stream))
    _raise(code, "kv_int4_attention")


def attention_noalloc(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, query_start_loc,
                      max_query_len, max_seq_len, softmax_scale, causal, signs, out,
                      dev_status: Optional[torch.Tensor] = None, stream=None, sliding_window: int = 0):
    """kv_int4_attention_noalloc: attention whose workspace is the library's
    static device scratch (for callers that cannot allocate device memory).

    Same arguments as attention() without ``workspace``.  Calls that overlap
    on the GPU share the scratch and race; issue them in order (one stream).
    Raises KvInt4Error(ERR_SCRATCH_LIMIT) when the sizes need more workspace
    than NOALLOC_SCRATCH_BYTES.
    """
    nb, bs, hkv, d = _cache_dims(k_cache, v_cache, k_scale, v_scale)
    _check(q.dim() == 3 and q.shape[2] == d, "q must be [tokens, q_heads, d]")
    hq = q.shape[1]
    qs = _token_major(q, "q", hq, d)
    os_ = _token_major(out, "out", hq, d)
    _check(out.shape[0] == q.shape[0], "out must match q")
    _check(block_table.dtype == torch.int32 and block_table.dim() == 2 and block_table.is_contiguous(),
           "block_table must be contiguous int32 [seqs, max_blocks]")
    _check(seq_lens.dtype == torch.int32 and query_start_loc.dtype == torch.int32, "seq_lens/query_start_loc int32")
    num_seqs = seq_lens.shape[0]
    _check(query_start_loc.shape[0] == num_seqs + 1 and block_table.shape[0] == num_seqs, "metadata shapes")
    _check(signs.dtype == torch.int8 and signs.numel() == d, "signs must be int8 [d]")
    lib = load()
    code = lib.kv_int4_attention_noalloc(_ptr(q), qs, _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                         _ptr(block_table), int(block_table.shape[1]), _ptr(seq_lens),
                                         _ptr(query_start_loc), int(num_seqs), int(q.shape[0]), int(max_query_len),
                                         int(max_seq_len), int(hq), int(hkv), int(d), int(bs), int(nb),
                                         float(softmax_scale), int(bool(causal)), int(sliding_window),
                                         _ptr(signs), _ptr(out), os_, _ptr(dev_status), _stream(stream))
    _raise(code, "kv_int4_attention_noalloc")


def attention_int8(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, query_start_loc,
                   max_query_len, max_seq_len, softmax_scale, causal, out, workspace,
                   dev_status: Optional[torch.Tensor] = None, stream=None, sliding_window: int = 0):
    """Attention over the int8_per_token_head cache through kv_int8_attention."""
    nb, bs, hkv, d = _cache_dims_int8(k_cache, v_cache, k_scale, v_scale)
    _check(q.dim() == 3 and q.shape[2] == d, "q must be [tokens, q_heads, d]")
    hq = q.shape[1]
    qs = _token_major(q, "q", hq, d)
    os_ = _token_major(out, "out", hq, d)
    _check(out.shape[0] == q.shape[0], "out must match q")
    _check(block_table.dtype == torch.int32 and block_table.dim() == 2 and block_table.is_contiguous(),
           "block_table must be contiguous int32 [seqs, max_blocks]")
    _check(seq_lens.dtype == torch.int32 and query_start_loc.dtype == torch.int32, "seq_lens/query_start_loc int32")
    num_seqs = seq_lens.shape[0]
    _check(query_start_loc.shape[0] == num_seqs + 1 and block_table.shape[0] == num_seqs, "metadata shapes")
    _check(workspace.dtype == torch.uint8 and workspace.is_contiguous(), "workspace must be contiguous uint8")
    code = load().kv_int8_attention(_ptr(q), qs, _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                    _ptr(block_table), int(block_table.shape[1]), _ptr(seq_lens),
                                    _ptr(query_start_loc), int(num_seqs), int(q.shape[0]), int(max_query_len),
                                    int(max_seq_len), int(hq), int(hkv), int(d), int(bs), int(nb),
                                    float(softmax_scale), int(bool(causal)), int(sliding_window), _ptr(out), os_,
                                    _ptr(workspace), int(workspace.numel()), _ptr(dev_status), _stream(stream))
    _raise(code, "kv_int8_attention")


def inslot_slot_bytes(head_size: int, int8: bool = False) -> int:
    """Bytes P of one (token, head) slot of the in-slot layout (0: unsupported head size)."""
    return int(load().kv_int4_inslot_slot_bytes(int(head_size), int(bool(int8))))


def _inslot_dims(kv_cache, head_size, int8):
    _check(kv_cache.dtype == torch.uint8 and kv_cache.dim() == 5 and kv_cache.shape[1] == 2 and
           kv_cache.is_contiguous(), "in-slot cache must be contiguous uint8 [blocks, 2, block_size, heads, P]")
    nb, _, bs, hkv, p = kv_cache.shape
    _check(p == inslot_slot_bytes(head_size, int8), f"slot bytes must be {inslot_slot_bytes(head_size, int8)}")
    return nb, bs, hkv


def write_inslot(k, v, slot_mapping, kv_cache, signs=None, int8: bool = False,
                 dev_status: Optional[torch.Tensor] = None, stream=None):
    """The INT4 (or int8_per_token_head) write into an in-slot cache."""
    d = k.shape[-1]
    nb, bs, hkv = _inslot_dims(kv_cache, d, int8)
    ks = _token_major(k, "k", hkv, d)
    vs = _token_major(v, "v", hkv, d)
    _check(k.shape[0] == v.shape[0] == slot_mapping.shape[0], "k, v and slot_mapping disagree on tokens")
    _check(slot_mapping.dtype == torch.int64 and slot_mapping.is_contiguous(), "slot_mapping must be contiguous int64")
    lib = load()
    if int8:
        code = lib.kv_int8_write_inslot(_ptr(k), ks, _ptr(v), vs, _ptr(slot_mapping), int(k.shape[0]),
                                        _ptr(kv_cache), nb, bs, hkv, d, _ptr(dev_status), _stream(stream))
    else:
        _check(signs is not None and signs.dtype == torch.int8 and signs.numel() == d, "signs must be int8 [d]")
        code = lib.kv_int4_write_inslot(_ptr(k), ks, _ptr(v), vs, _ptr(slot_mapping), int(k.shape[0]),
                                        _ptr(kv_cache), nb, bs, hkv, d, _ptr(signs), _ptr(dev_status),
                                        _stream(stream))
    _raise(code, "kv_int8_write_inslot" if int8 else "kv_int4_write_inslot")


def attention_inslot(q, kv_cache, block_table, seq_lens, query_start_loc, max_query_len, max_seq_len,
                     softmax_scale, causal, out, workspace, signs=None, int8: bool = False,
                     dev_status: Optional[torch.Tensor] = None, stream=None, sliding_window: int = 0):
    """Attention over an in-slot INT4 (or int8_per_token_head) cache."""
    _check(q.dim() == 3, "q must be [tokens, q_heads, d]")
    hq, d = q.shape[1], q.shape[2]
    nb, bs, hkv = _inslot_dims(kv_cache, d, int8)
    qs = _token_major(q, "q", hq, d)
    os_ = _token_major(out, "out", hq, d)
    _check(out.shape[0] == q.shape[0], "out must match q")
    _check(block_table.dtype == torch.int32 and block_table.dim() == 2 and block_table.is_contiguous(),
           "block_table must be contiguous int32 [seqs, max_blocks]")
    num_seqs = seq_lens.shape[0]
    _check(query_start_loc.shape[0] == num_seqs + 1 and block_table.shape[0] == num_seqs, "metadata shapes")
    _check(workspace.dtype == torch.uint8 and workspace.is_contiguous(), "workspace must be contiguous uint8")
    lib = load()
    common = (_ptr(q), qs, _ptr(kv_cache), _ptr(block_table), int(block_table.shape[1]), _ptr(seq_lens),
              _ptr(query_start_loc), int(num_seqs), int(q.shape[0]), int(max_query_len), int(max_seq_len), int(hq),
              int(hkv), int(d), int(bs), int(nb), float(softmax_scale), int(bool(causal)), int(sliding_window))
    tail = (_ptr(out), os_, _ptr(workspace), int(workspace.numel()), _ptr(dev_status), _stream(stream))
    if int8:
        code = lib.kv_int8_attention_inslot(*common, *tail)
    else:
        _check(signs is not None and signs.dtype == torch.int8 and signs.numel() == d, "signs must be int8 [d]")
        code = lib.kv_int4_attention_inslot(*common, _ptr(signs), *tail)
    _raise(code, "kv_int8_attention_inslot" if int8 else "kv_int4_attention_inslot")
