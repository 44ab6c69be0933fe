"""Plain fp64 CPU oracle for the INT4 per-token-head KV cache with a randomized
Hadamard rotation (RHT) and for paged attention over that cache.

TEST INFRASTRUCTURE ONLY.  This module is imported by the tests, by
``__graft_entry__.smoke()`` and by the CPU-baseline leg of ``bench.py``; the
library's product path never imports or calls it.  It shares no code, tables
or constants with the CUDA path.

What it follows (sources are the method's pages):

* "Rotate KV into RHT domain in the INT4 unified attn test" (vLLM PR #62881),
  section Details / Root cause: the write path stores K_s = H.D.k with D a
  random +-1 diagonal (D.D = I) and H a Walsh-Hadamard matrix; the read path
  rotates q' = H.D.q, scales scores by softmax_scale/d so that q'.K_s/d = q.k,
  and applies D.H(.)/d to the output to undo V's rotation.  Section Details /
  Fix: the rotation is rounded through bf16 before quantisation.
* "vLLM -- Attention Kernels & KV Cache Quantization" (PR #56198, section
  "Merged contribution"): for d = b.n with b the largest power-of-two divisor
  of d, H_b is applied block-diagonally inside each of the n blocks; H.H^T =
  b.I, and every 1/d compensation above becomes 1/b.
* "[Feature] Triton INT4 per-token-head KV cache quantization" (vLLM PR
  #40835), review thread: caches are [num_blocks, block_size, num_kv_heads,
  d/2] uint8 with f32 scale caches [num_blocks, block_size, num_kv_heads],
  written through slot_mapping; block = slot // block_size, offset = slot %
  block_size.

Readings taken where the pages are silent (each is also listed in the design
notes): scale = fp32(absmax / 7) (symmetric, codes in [-7, 7], clamp to
[-8, 7] as a guard); code = round-half-even(y * r) with r the fp32-rounded
reciprocal of the stored scale and the product taken exactly; a vector whose
absmax is below 2^-120 is stored as scale 0 and all-zero codes; element 2j of
a head vector goes to the low nibble of byte j and element 2j+1 to the high
nibble, in 4-bit two's complement; H_b is the Sylvester (natural-order)
matrix with entries (-1)^popcount(i & j); D is applied before H.

Parity pins: every function here is pinned by tests in ``tests/`` against
scipy's Hadamard construction, closed forms, hand-derived worked examples
(``tests/golden/``), brute-force loops and the pages' published error bounds.
The nibble order, the scale divisor and D's generator are this library's
definitions (the pages print no worked example with values for them): those
three points are pinned only by the hand-derived fixtures that define them.
"""

from __future__ import annotations

import numpy as np

BF16_MAX = float.fromhex("0x1.fep127")
# Below this absmax a vector is stored as scale 0 / codes 0 (see module doc).
FLUSH_ABSMAX = 2.0 ** -120


# ---------------------------------------------------------------------------
# Rotation
# ---------------------------------------------------------------------------

def largest_pow2_divisor(d: int) -> int:
    """b = the largest power of two dividing d (PR #56198 page)."""
    if d <= 0:
        raise ValueError("head size must be positive")
    b = 1
    while d % (2 * b) == 0:
        b *= 2
    return b


def hadamard(b: int) -> np.ndarray:
    """Unnormalised Sylvester Walsh-Hadamard matrix, H[i, j] = (-1)^popcount(i & j)."""
    if b <= 0 or b & (b - 1):
        raise ValueError("Hadamard order must be a power of two")
    i = np.arange(b)
    bits = np.bitwise_and.outer(i, i)
    parity = np.zeros_like(bits)
    while bits.any():
        parity ^= bits & 1
        bits >>= 1
    return np.where(parity == 1, -1.0, 1.0)


def block_hadamard(d: int) -> np.ndarray:
    """I_n (x) H_b: H_b on each contiguous block [j*b, (j+1)*b) of a head vector."""
    b = largest_pow2_divisor(d)
    return np.kron(np.eye(d // b), hadamard(b))


def rht_forward(x, signs) -> np.ndarray:
    """y = (I_n (x) H_b) . D . x over the last axis, in fp64 (no rounding)."""
    x = np.asarray(x, dtype=np.float64)
    s = np.asarray(signs, dtype=np.float64)
    hb = block_hadamard(x.shape[-1])
    return (x * s) @ hb.T


def rht_inverse(y, signs) -> np.ndarray:
    """x = D . (I_n (x) H_b) . y / b over the last axis, in fp64."""
    y = np.asarray(y, dtype=np.float64)
    d = y.shape[-1]
    b = largest_pow2_divisor(d)
    hb = block_hadamard(d)
    return (y @ hb.T) * np.asarray(signs, dtype=np.float64) / b


# ---------------------------------------------------------------------------
# bf16 rounding (round to nearest, ties to even, directly from fp64)
# ---------------------------------------------------------------------------

def round_bf16(x) -> np.ndarray:
    """Round fp64 values to the nearest bf16 value (ties to even), as fp64.

    bf16 keeps 8 significant bits and fp32's exponent range; subnormals are
    spaced 2^-133 apart.  Values beyond the largest finite bf16 after
    rounding become +-inf.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, copy=True)
    finite = np.isfinite(x) & (x != 0)
    xf = x[finite]
    _, e = np.frexp(xf)                       # |x| in [2^(e-1), 2^e)
    e = np.maximum(e, -125)                   # bf16 normals start at 2^-126
    quantum = np.ldexp(1.0, e - 8)
    r = np.rint(xf / quantum) * quantum       # np.rint rounds half to even
    r = np.where(np.abs(r) > BF16_MAX, np.copysign(np.inf, r), r)
    out[finite] = r
    return out


# ---------------------------------------------------------------------------
# Quantiser and packing
# ---------------------------------------------------------------------------

def quantize(y_bf16):
    """Per-vector absmax INT4 quantisation over the last axis.

    Returns (codes int8 [..., d] in [-8, 7], scale float32 [...]).
      a = max_i |y_i|                                     (exact)
      s = fp32(a / 7)         IEEE fp32 division            (stored scale)
      r = fp32(1 / s)         IEEE fp32 reciprocal
      c = clamp(round_half_even(y * r), -8, 7), y*r exact in fp64
    with s = 0, c = 0 when a < 2^-120.
    """
    y = np.asarray(y_bf16, dtype=np.float64)
    a = np.max(np.abs(y), axis=-1)
    a32 = a.astype(np.float32)                 # a is a bf16 value: exact
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        s = (a32 / np.float32(7.0)).astype(np.float32)
        r = (np.float32(1.0) / s).astype(np.float32)
    flush = a < FLUSH_ABSMAX
    s = np.where(flush, np.float32(0.0), s).astype(np.float32)
    r = np.where(flush, np.float32(0.0), r).astype(np.float32)
    prod = y * r.astype(np.float64)[..., None]  # 8-bit x 24-bit significands: exact
    c = np.clip(np.rint(prod), -8, 7).astype(np.int8)
    return c, s


def pack_codes(codes) -> np.ndarray:
    """Two 4-bit two's-complement codes per byte: element 2j low, 2j+1 high."""
    c = np.asarray(codes).astype(np.int16)
    nib = (c & 0xF).astype(np.uint8)
    return (nib[..., 0::2] | (nib[..., 1::2] << 4)).astype(np.uint8)


def unpack_codes(packed) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    lo = (p & 0xF).astype(np.int16)
    hi = (p >> 4).astype(np.int16)
    lo = np.where(lo >= 8, lo - 16, lo)
    hi = np.where(hi >= 8, hi - 16, hi)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.int8)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


# ---------------------------------------------------------------------------
# Write path (reshape_and_cache_int4)
# ---------------------------------------------------------------------------

def rotate_for_cache(x, signs) -> np.ndarray:
    """bf16(H_b-blockdiag . D . x): the rotated value that gets quantised."""
    return round_bf16(rht_forward(x, signs))


def write_cache(k, v, slot_mapping, k_cache, v_cache, k_scale, v_scale,
                block_size, signs=None, prerotated=False):
    """Quantise new K/V head vectors and scatter them into the paged cache.

    k, v: [T, Hkv, d] values (fp64 or anything convertible; bf16 inputs are
    exact).  Caches are updated in place: k_cache/v_cache uint8 [NB, bs, Hkv,
    d/2], k_scale/v_scale float32 [NB, bs, Hkv].  Tokens with slot < 0 are
    skipped.  With ``prerotated`` the inputs are already the bf16 rotated
    values and the rotation is not applied.  Returns the set of slots that
    were outside [0, NB*bs) (and skipped).
    """
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    slots = np.asarray(slot_mapping, dtype=np.int64)
    nb = k_cache.shape[0]
    bad = []
    if prerotated:
        ky, vy = k, v
    else:
        ky = rotate_for_cache(k, signs)
        vy = rotate_for_cache(v, signs)
    kc, ks = quantize(ky)
    vc, vs = quantize(vy)
    kp = pack_codes(kc)
    vp = pack_codes(vc)
    for t, slot in enumerate(slots):
        if slot < 0:
            continue
        if slot >= nb * block_size:
            bad.append(int(slot))
            continue
        blk, off = divmod(int(slot), block_size)
        k_cache[blk, off] = kp[t]
        v_cache[blk, off] = vp[t]
        k_scale[blk, off] = ks[t]
        v_scale[blk, off] = vs[t]
    return bad


# ---------------------------------------------------------------------------
# Read path (unified_attention_int4), plain definition in the original domain
# ---------------------------------------------------------------------------

def gather_sequence(cache, scale, block_table_row, seq_len, kv_head, block_size):
    """Codes [L, d] (int8) and scales [L] (fp64) of positions 0..L-1 of one head."""
    pos = np.arange(seq_len)
    blk = np.asarray(block_table_row, dtype=np.int64)[pos // block_size]
    off = pos % block_size
    codes = unpack_codes(cache[blk, off, kv_head])
    s = scale[blk, off, kv_head].astype(np.float64)
    return codes, s


def dequantize_original(codes, scales, signs) -> np.ndarray:
    """k_hat = D . (I_n (x) H_b) . (c * s) / b : the cache entry in the original domain."""
    rot = np.asarray(codes, dtype=np.float64) * np.asarray(scales, dtype=np.float64)[..., None]
    return rht_inverse(rot, signs)


def attention_head(q_rows, k_hat, v_hat, ctx, softmax_scale, causal, sliding_window=0):
    """softmax(scale * q k^T + mask) v for one q head of one sequence, fp64.

    q_rows [q_len, d]; k_hat, v_hat [L, d]; query j sits at position ctx + j
    and, when causal, sees keys 0..ctx+j; otherwise all L keys.  A sliding
    window W > 0 also hides every key t with (ctx + j) - t >= W, i.e. the
    query keeps the W positions ending at its own (the "added window" of the
    Triton INT4 PR, read with vLLM's window rule).
    """
    q = np.asarray(q_rows, dtype=np.float64)
    scores = softmax_scale * (q @ k_hat.T)
    L = k_hat.shape[0]
    j = np.arange(q.shape[0])[:, None]
    t = np.arange(L)[None, :]
    if causal:
        scores = np.where(t <= ctx + j, scores, -np.inf)
    if sliding_window > 0:
        scores = np.where((ctx + j) - t < sliding_window, scores, -np.inf)
    m = np.max(scores, axis=1, keepdims=True)
    p = np.exp(scores - m)
    p /= np.sum(p, axis=1, keepdims=True)
    return p @ v_hat


def attention_seq(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens,
                  query_start_loc, seq, num_kv_heads, block_size, softmax_scale,
                  causal, signs, q_heads=None, sliding_window=0):
    """Output rows [q_len, Hq, d] (fp64) of one sequence; optionally only some q heads.

    q is [num_q_tokens, Hq, d]; q head h uses kv head h // (Hq / Hkv).
    """
    q = np.asarray(q)
    hq = q.shape[1]
    d = q.shape[2]
    group = hq // num_kv_heads
    q0, q1 = int(query_start_loc[seq]), int(query_start_loc[seq + 1])
    L = int(seq_lens[seq])
    ctx = L - (q1 - q0)
    heads = range(hq) if q_heads is None else q_heads
    out = np.zeros((q1 - q0, hq, d))
    cache_rows = {}
    for h in heads:
        kvh = h // group
        if kvh not in cache_rows:
            kc, ks = gather_sequence(k_cache, k_scale, block_table[seq], L, kvh, block_size)
            vc, vs = gather_sequence(v_cache, v_scale, block_table[seq], L, kvh, block_size)
            cache_rows[kvh] = (dequantize_original(kc, ks, signs),
                               dequantize_original(vc, vs, signs))
        k_hat, v_hat = cache_rows[kvh]
        out[:, h, :] = attention_head(q[q0:q1, h, :], k_hat, v_hat, ctx, softmax_scale, causal,
                                      sliding_window)
    return out


def attention(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens,
              query_start_loc, num_kv_heads, block_size, softmax_scale, causal, signs,
              sliding_window=0):
    """Full attention output [num_q_tokens, Hq, d] in fp64, streamed per sequence."""
    q = np.asarray(q)
    out = np.zeros(q.shape, dtype=np.float64)
    for s in range(len(seq_lens)):
        q0, q1 = int(query_start_loc[s]), int(query_start_loc[s + 1])
        if q1 == q0:
            continue
        out[q0:q1] = attention_seq(q, k_cache, v_cache, k_scale, v_scale, block_table,
                                   seq_lens, query_start_loc, s, num_kv_heads, block_size,
                                   softmax_scale, causal, signs, sliding_window=sliding_window)
    return out


def rotated_domain_scores(q_rows, codes, scales, signs, softmax_scale):
    """The read path's own score formula: (softmax_scale / b) * q' . (c * s).

    Used by the tests to pin that the rotated-domain computation equals the
    original-domain one (q'.K_s/b = q.k).
    """
    d = codes.shape[-1]
    b = largest_pow2_divisor(d)
    qr = rht_forward(q_rows, signs)
    rot = np.asarray(codes, dtype=np.float64) * np.asarray(scales, dtype=np.float64)[..., None]
    return (softmax_scale / b) * (qr @ rot.T)


# ---------------------------------------------------------------------------
# Sibling mode: int8_per_token_head ("[Feature] Triton INT4 per-token-head KV
# cache quantization", PR #40835, review thread: the int8 cache dtype, the
# raw-cache "round reference" test, the 0.1 dequantisation tolerance;
# "vLLM -- Attention Kernels & KV Cache Quantization", Merged contribution:
# int8_per_token_head never uses the transform).  Readings: scale =
# fp32(absmax / 127) (symmetric, codes in [-127, 127], clamp to [-128, 127]
# as a guard), code = round-half-even(x * r) with r = fp32(1 / s) and the
# product exact, the same evaluation as the INT4 mode; vectors with absmax
# below 2^-119 (where absmax / 127 would leave the fp32 normal range) are
# stored as scale 0 and zero codes.  Caches: int8 [NB, bs, Hkv, d], scales
# float32 [NB, bs, Hkv].
# ---------------------------------------------------------------------------

FLUSH_ABSMAX_INT8 = 2.0 ** -119


def quantize_int8(x_bf16):
    """Per-vector absmax INT8 quantisation over the last axis, no rotation.

    Returns (codes int8 [..., d] in [-128, 127], scale float32 [...]).
      a = max_i |x_i|;  s = fp32(a / 127);  r = fp32(1 / s)
      c = clamp(round_half_even(x * r), -128, 127), x*r exact in fp64
    with s = 0, c = 0 when a < 2^-119.
    """
    x = np.asarray(x_bf16, dtype=np.float64)
    a = np.max(np.abs(x), axis=-1)
    a32 = a.astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        s = (a32 / np.float32(127.0)).astype(np.float32)
        r = (np.float32(1.0) / s).astype(np.float32)
    flush = a < FLUSH_ABSMAX_INT8
    s = np.where(flush, np.float32(0.0), s).astype(np.float32)
    r = np.where(flush, np.float32(0.0), r).astype(np.float32)
    prod = x * r.astype(np.float64)[..., None]
    c = np.clip(np.rint(prod), -128, 127).astype(np.int8)
    return c, s


def write_cache_int8(k, v, slot_mapping, k_cache, v_cache, k_scale, v_scale, block_size):
    """Quantise new K/V head vectors (no rotation) into the int8 paged cache.

    k, v: [T, Hkv, d]; k_cache/v_cache int8 [NB, bs, Hkv, d], scales float32
    [NB, bs, Hkv], updated in place; slot < 0 skipped; returns the slots that
    were outside [0, NB*bs) (and skipped)."""
    kc, ks = quantize_int8(k)
    vc, vs = quantize_int8(v)
    nb = k_cache.shape[0]
    bad = []
    for t, slot in enumerate(np.asarray(slot_mapping, dtype=np.int64)):
        if slot < 0:
            continue
        if slot >= nb * block_size:
            bad.append(int(slot))
            continue
        blk, off = divmod(int(slot), block_size)
        k_cache[blk, off] = kc[t]
        v_cache[blk, off] = vc[t]
        k_scale[blk, off] = ks[t]
        v_scale[blk, off] = vs[t]
    return bad


def attention_int8(q, k_cache, v_cache, k_scale, v_scale, block_table, seq_lens, query_start_loc,
                   num_kv_heads, block_size, softmax_scale, causal, sliding_window=0):
    """Attention over the int8 cache: k_hat = c * s (no rotation), then the
    same softmax(scale * q k_hat^T + mask) v_hat per q head as the INT4 mode."""
    q = np.asarray(q, dtype=np.float64)
    hq = q.shape[1]
    group = hq // num_kv_heads
    out = np.zeros(q.shape, dtype=np.float64)
    for s in range(len(seq_lens)):
        q0, q1 = int(query_start_loc[s]), int(query_start_loc[s + 1])
        if q1 == q0:
            continue
        L = int(seq_lens[s])
        pos = np.arange(L)
        blk = np.asarray(block_table[s], dtype=np.int64)[pos // block_size]
        off = pos % block_size
        for h in range(hq):
            kvh = h // group
            k_hat = k_cache[blk, off, kvh].astype(np.float64) * k_scale[blk, off, kvh].astype(np.float64)[:, None]
            v_hat = v_cache[blk, off, kvh].astype(np.float64) * v_scale[blk, off, kvh].astype(np.float64)[:, None]
            out[q0:q1, h] = attention_head(q[q0:q1, h], k_hat, v_hat, L - (q1 - q0), softmax_scale, causal,
                                           sliding_window)
    return out


# ---------------------------------------------------------------------------
# In-slot scale layout ("[Feature] Triton INT4 per-token-head KV cache
# quantization", PR #40835, review thread: a block holds a K half then a V
# half, each (token, head) slot padded_hs wide with the f32 scale at offset hs
# inside it; #62113 per "Rotate KV into RHT domain in the INT4 unified attn
# test", Validation: 16-byte-aligned slots).  Reading: slot bytes P =
# round_up(CB + 4, 16) with CB code bytes per head vector; codes at [0, CB),
# the scale at [CB, CB + 4), padding after; cache uint8 [NB, 2, bs, Hkv, P].
# A re-arrangement only: the values are those of the separate caches.
# ---------------------------------------------------------------------------

def inslot_slot_bytes(code_bytes: int) -> int:
    return (code_bytes + 4 + 15) // 16 * 16


def to_inslot(k_cache, v_cache, k_scale, v_scale, fill=0):
    """The combined in-slot cache holding the given separate caches' codes and
    scales (padding bytes = fill)."""
    kc = np.asarray(k_cache).view(np.uint8)
    vc = np.asarray(v_cache).view(np.uint8)
    nb, bs, hkv, cb = kc.shape
    P = inslot_slot_bytes(cb)
    out = np.full((nb, 2, bs, hkv, P), fill, dtype=np.uint8)
    out[:, 0, :, :, :cb] = kc
    out[:, 1, :, :, :cb] = vc
    out[:, 0, :, :, cb:cb + 4] = np.ascontiguousarray(np.asarray(k_scale, np.float32)).view(np.uint8).reshape(
        nb, bs, hkv, 4)
    out[:, 1, :, :, cb:cb + 4] = np.ascontiguousarray(np.asarray(v_scale, np.float32)).view(np.uint8).reshape(
        nb, bs, hkv, 4)
    return out


def from_inslot(cache, code_bytes):
    """Separate (k_cache, v_cache, k_scale, v_scale) views of an in-slot cache."""
    c = np.asarray(cache, dtype=np.uint8)
    cb = code_bytes
    kc = np.ascontiguousarray(c[:, 0, :, :, :cb])
    vc = np.ascontiguousarray(c[:, 1, :, :, :cb])
    ks = np.ascontiguousarray(c[:, 0, :, :, cb:cb + 4]).view(np.float32)[..., 0]
    vs = np.ascontiguousarray(c[:, 1, :, :, cb:cb + 4]).view(np.float32)[..., 0]
    return kc, vc, ks, vs
