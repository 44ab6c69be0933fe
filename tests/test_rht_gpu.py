"""Parity of kv_int4_rht (CUDA, through the C ABI) with the fp64 oracle's
rht_forward / rht_inverse: the block-diagonal randomized Hadamard rotation
of "vLLM -- Attention Kernels & KV Cache Quantization" (Merged contribution),
D applied first as in "Rotate KV into RHT domain in the INT4 unified attn
test" (Details / Root cause)."""

import numpy as np
import pytest
import torch

from oracle import kvint4_oracle as O
from int4_token_head_gb300 import _lib
from tests.helpers import f32_bits

pytestmark = pytest.mark.gpu
REG_HEADS = [64, 96, 128, 192, 256]                       # register kernel
SMEM_HEADS = [1, 2, 3, 6, 10, 33, 48, 80, 112, 160, 320, 1000, 4096]  # shared-memory kernel


def _signs(d, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randint(0, 2, (d,), generator=g) * 2 - 1).to(torch.int8)


def _ints(rows, d, lo, hi, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, (rows, d), generator=g).to(torch.bfloat16)


@pytest.mark.parametrize("d", REG_HEADS + SMEM_HEADS)
@pytest.mark.parametrize("inverse", [False, True])
def test_rht_bit_exact_on_integer_inputs(d, inverse):
    """Small integers keep every fp32 partial sum exact (|sum| <= 64 * 4096 <
    2^24) and /b is a power of two, so fp32 results equal the fp64 oracle and
    the bf16 results equal its single rounding."""
    rows = 37 if d <= 1000 else 5
    x = _ints(rows, d, -64, 64, d + 7 * inverse)
    s = _signs(d, d)
    ref = (O.rht_inverse if inverse else O.rht_forward)(x.double().numpy(), s.numpy())
    y32 = _lib.rht(x.cuda(), s.cuda(), inverse=inverse, out_dtype=torch.float32).cpu().numpy()
    assert np.array_equal(y32.astype(np.float64), ref)
    y16 = _lib.rht(x.cuda(), s.cuda(), inverse=inverse).float().cpu().numpy()
    assert np.array_equal(y16.astype(np.float64), O.round_bf16(ref))


@pytest.mark.parametrize("d", REG_HEADS + [6, 80, 320])
def test_rht_random_inputs_within_the_fp32_butterfly_bound(d):
    """N(0,1) inputs: each of the log2(b) butterfly stages rounds once, and
    every partial sum is bounded by the block's L1 norm, so
    |y - y_exact| <= log2(b) * 2^-24 * max_block ||x||_1."""
    rows = 300
    g = torch.Generator().manual_seed(d)
    x = torch.randn((rows, d), generator=g).to(torch.bfloat16)
    s = _signs(d, d + 1)
    xd = x.double().numpy()
    b = O.largest_pow2_divisor(d)
    l1 = np.abs(xd).reshape(rows, d // b, b).sum(axis=2).max(axis=1)
    stages = max(1, int(np.log2(b)))
    for inverse, scale in ((False, 1.0), (True, 1.0 / b)):
        ref = (O.rht_inverse if inverse else O.rht_forward)(xd, s.numpy())
        got = _lib.rht(x.cuda(), s.cuda(), inverse=inverse, out_dtype=torch.float32).double().cpu().numpy()
        bound = stages * 2.0 ** -24 * l1 * scale * 1.0001
        assert np.all(np.abs(got - ref).max(axis=1) <= bound), (d, inverse)


@pytest.mark.parametrize("d", REG_HEADS + [6, 48, 1000])
def test_rht_round_trip_is_exact_on_sparse_sign_vectors(d):
    """x with at most 8 nonzero +-1 entries per Hadamard block: y = rht(x) has
    |y| <= 8 (bf16 exact), so rht(y, inverse) returns x exactly."""
    rows = 64
    g = torch.Generator().manual_seed(3 * d)
    b = O.largest_pow2_divisor(d)
    x = torch.zeros((rows, d))
    for r in range(rows):
        for blk in range(d // b):
            idx = torch.randperm(b, generator=g)[:min(8, b)] + blk * b
            x[r, idx] = (torch.randint(0, 2, (len(idx),), generator=g) * 2 - 1).float()
    x = x.to(torch.bfloat16).cuda()
    s = _signs(d, 5).cuda()
    y = _lib.rht(x, s)
    back = _lib.rht(y, s, inverse=True)
    assert torch.equal(back, x)


def test_rht_strided_rows_and_output_view():
    """Rows taken from a wider tensor (a K slice of a fused qkv layout) and an
    output written into a slice of a larger fp32 buffer; nothing outside is
    touched."""
    d, rows = 128, 200
    g = torch.Generator().manual_seed(11)
    qkv = torch.randn((rows, 3 * d), generator=g).to(torch.bfloat16).cuda()
    x = qkv[:, d:2 * d]
    s = _signs(d, 12).cuda()
    big = torch.full((rows, 2 * d), 7.0, dtype=torch.float32, device="cuda")
    out = big[:, :d]
    _lib.rht(x, s, out=out)
    ref = O.rht_forward(x.double().cpu().numpy(), s.cpu().numpy())
    assert np.abs(out.double().cpu().numpy() - ref).max() < 1e-3
    assert torch.all(big[:, d:] == 7.0)


def test_rht_batch_of_a_write_chunk_matches_sampled_rows():
    """The bench's size: a 65,536-token x 8-head K chunk (d=128), sampled
    rows against the oracle within the fp32 bound; empty batch enqueues
    nothing."""
    d, rows = 128, 65536 * 8
    g = torch.Generator(device="cuda").manual_seed(5)
    x = torch.randn((rows, d), generator=g, device="cuda").to(torch.bfloat16)
    s = _signs(d, 6).cuda()
    y = _lib.rht(x, s, out_dtype=torch.float32)
    idx = torch.randint(0, rows, (512,), generator=torch.Generator().manual_seed(1))
    xs = x[idx.cuda()].double().cpu().numpy()
    ref = O.rht_forward(xs, s.cpu().numpy())
    bound = 7 * 2.0 ** -24 * np.abs(xs).sum(axis=1) * 1.0001
    assert np.all(np.abs(y[idx.cuda()].double().cpu().numpy() - ref).max(axis=1) <= bound)
    empty = torch.empty((0, d), dtype=torch.bfloat16, device="cuda")
    assert _lib.rht(empty, s).shape == (0, d)


@pytest.mark.parametrize("d", REG_HEADS)
def test_rht_unaligned_rows_take_the_scalar_kernel(d):
    """Rows starting 2 bytes past a 16-byte boundary (and an output 4 bytes
    off) are served by the one-row-per-warp kernel: same exact results."""
    rows = 70
    buf = _ints(rows, d + 8, -64, 64, d + 100).cuda()
    x = buf[:, 1:1 + d]
    s = _signs(d, d + 3)
    ref = O.rht_forward(x.double().cpu().numpy(), s.numpy())
    obuf = torch.zeros((rows, d + 4), dtype=torch.float32, device="cuda")
    out = obuf[:, 1:1 + d]
    _lib.rht(x, s.cuda(), out=out)
    assert np.array_equal(out.double().cpu().numpy(), ref)
    assert torch.all(obuf[:, 0] == 0) and torch.all(obuf[:, 1 + d:] == 0)
    ref_inv = O.rht_inverse(x.double().cpu().numpy(), s.numpy())
    got_inv = _lib.rht(x, s.cuda(), inverse=True).float().cpu().numpy()
    assert np.array_equal(got_inv.astype(np.float64), O.round_bf16(ref_inv))
