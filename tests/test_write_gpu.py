"""Parity of kv_int4_write (CUDA, through the C ABI) with the fp64 oracle."""

import numpy as np
import pytest
import torch

from oracle import kvint4_oracle as O
from int4_token_head_gb300 import _lib, synthetic
from tests.helpers import f32_bits

pytestmark = pytest.mark.gpu
HEADS = [64, 96, 128, 192, 256]


def _empty(nb, hkv, d, dev="cuda"):
    w = synthetic.custom_workload(hkv, hkv, d, [(1, 1)])
    w.num_blocks = nb
    return w.empty_cache(dev)


def _run_gpu_write(k, v, slots, nb, signs, prerotated=False, stream_k=None):
    hkv, d = k.shape[1], k.shape[2]
    kc, vc, ks, vs = _empty(nb, hkv, d)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _lib.write(k.cuda() if stream_k is None else stream_k, v.cuda(), slots.cuda(), kc, vc, ks, vs,
               signs.cuda(), dev_status=status, prerotated=prerotated)
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in (kc, vc, ks, vs)], int(status.item())


def _oracle_write(k, v, slots, nb, signs, prerotated=False):
    hkv, d = k.shape[1], k.shape[2]
    caches = [t.numpy() for t in _empty(nb, hkv, d, "cpu")]
    O.write_cache(k.float().numpy(), v.float().numpy(), slots.numpy(), *caches, 16,
                  signs.numpy(), prerotated=prerotated)
    return caches


def _signs(d, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randint(0, 2, (d,), generator=g) * 2 - 1).to(torch.int8)


def _rotated_inputs(T, hkv, d, seed):
    """bf16 rotated values y = oracle rotation of random inputs, plus special rows."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((T, hkv, d), generator=g).to(torch.bfloat16)
    y = O.rotate_for_cache(x.double().numpy(), _signs(d, seed + 1).numpy().astype(np.float64))
    y = torch.from_numpy(y).to(torch.bfloat16)
    y[0, 0] = 0                                     # zero vector: scale 0, codes 0
    y[1, 0] = (y[1, 0].double() * 1e-38).to(torch.bfloat16)  # below the flush bound
    # exact ties: absmax 7 (scale 1, reciprocal 1) and half-integer entries
    tie = torch.tensor([(i % 15) - 7 + (0.5 if i % 3 == 0 else 0.0) for i in range(d)]).clamp(-6.5, 6.5)
    tie[5] = 7.0
    y[2, 0] = tie.to(torch.bfloat16)
    return y


@pytest.mark.parametrize("d", HEADS)
def test_prerotated_codes_and_scales_bit_exact(d):
    T, hkv, nb = 357, 4, 100  # ragged against every tile size
    ky = _rotated_inputs(T, hkv, d, 10 + d)
    vy = _rotated_inputs(T, hkv, d, 20 + d)
    g = torch.Generator().manual_seed(d)
    slots = torch.randperm(nb * 16, generator=g)[:T].to(torch.int64)
    slots[7] = -1  # padding token
    got, status = _run_gpu_write(ky, vy, slots, nb, _signs(d, 0), prerotated=True)
    ref = _oracle_write(ky, vy, slots, nb, _signs(d, 0), prerotated=True)
    assert status == 0
    for a, b, name in zip(got, ref, ["k_cache", "v_cache", "k_scale", "v_scale"]):
        if a.dtype == np.float32:
            assert np.array_equal(f32_bits(a), f32_bits(b)), name
        else:
            assert np.array_equal(a, b), name


@pytest.mark.parametrize("d", [64, 96, 128, 192])
def test_write_scale_and_codes_exact_over_all_absmax_mantissas(d):
    """Head vectors with a single nonzero entry c: every rotated element is
    +-c exactly (on both sides), so the absmax is |c| and the scale must be
    fp32(|c| / 7) bit for bit, with codes +-7.  c sweeps all 128 bf16
    mantissas over exponents from below the flush bound (2^-120) to 2^126."""
    hkv = 4
    exps = [-121, -120, -119, -100, -30, -1, 0, 1, 7, 40, 100, 126]
    vals = np.array([(1 + m / 128) * 2.0 ** e * (1 if (m + e) % 2 else -1) for e in exps for m in range(128)])
    n = len(vals)
    T = (n + hkv - 1) // hkv
    g = torch.Generator().manual_seed(d)
    k = torch.zeros((T, hkv, d), dtype=torch.float64)
    v = torch.zeros((T, hkv, d), dtype=torch.float64)
    perm = torch.randperm(n, generator=g).numpy()
    for u in range(T * hkv):
        t, h = divmod(u, hkv)
        k[t, h, (7 * u + 3) % d] = float(vals[u % n])
        v[t, h, (5 * u + 1) % d] = float(vals[perm[u % n]])
    k, v = k.to(torch.bfloat16), v.to(torch.bfloat16)
    assert np.array_equal(k.double().numpy().sum(axis=2).ravel()[:n], vals)  # every c is a bf16 value
    nb = (T + 15) // 16 + 3
    slots = torch.randperm(nb * 16, generator=g)[:T].to(torch.int64)
    signs = _signs(d, 5)
    got, status = _run_gpu_write(k, v, slots, nb, signs)
    ref = _oracle_write(k, v, slots, nb, signs)
    assert status == 0
    for a, b, name in zip(got, ref, ["k_cache", "v_cache", "k_scale", "v_scale"]):
        if a.dtype == np.float32:
            assert np.array_equal(f32_bits(a), f32_bits(b)), name
        else:
            assert np.array_equal(a, b), name


@pytest.mark.parametrize("d", HEADS)
def test_write_end_to_end_within_one_code(d):
    """Raw bf16 K/V -> rotation in fp32 on the GPU vs fp64 in the oracle:
    slots and untouched bytes bit-exact, codes within +-1, scales within one
    bf16 ulp of absmax / 7."""
    T, hkv, nb = 1000, 8, 600
    g = torch.Generator().manual_seed(100 + d)
    k = (torch.randn((T, hkv, d), generator=g) * 2).to(torch.bfloat16)
    v = torch.randn((T, hkv, d), generator=g).to(torch.bfloat16)
    signs = _signs(d, d)
    slots = torch.randperm(nb * 16, generator=g)[:T].to(torch.int64)
    slots[::97] = -1
    got, status = _run_gpu_write(k, v, slots, nb, signs)
    ref = _oracle_write(k, v, slots, nb, signs)
    assert status == 0
    written = np.zeros(nb * 16, bool)
    written[slots[slots >= 0].numpy()] = True
    written = written.reshape(nb, 16)
    for which in (0, 1):
        gc, rc = got[which], ref[which]
        gs, rs = got[2 + which], ref[2 + which]
        # untouched slots keep the sentinels bit for bit
        assert np.array_equal(gc[~written], rc[~written])
        assert np.array_equal(f32_bits(gs[~written]), f32_bits(rs[~written]))
        gcodes = O.unpack_codes(gc[written]).astype(np.int32)
        rcodes = O.unpack_codes(rc[written]).astype(np.int32)
        diff = np.abs(gcodes - rcodes)
        assert diff.max() <= 1
        assert diff.mean() < 1e-3
        rel = np.abs(gs[written].astype(np.float64) - rs[written]) / rs[written]
        assert rel.max() <= 2.0 ** -7  # one bf16 ulp of absmax, carried into absmax/7
        assert np.mean(rel == 0) > 0.99


def test_write_strided_qkv_view_and_edge_slots():
    d, hkv, hq, nb = 128, 8, 32, 20
    T = 77
    g = torch.Generator().manual_seed(5)
    qkv = torch.randn((T, (hq + 2 * hkv) * d), generator=g).to(torch.bfloat16)
    k = qkv[:, hq * d:(hq + hkv) * d].view(T, hkv, d)
    v = qkv[:, (hq + hkv) * d:].view(T, hkv, d)
    assert k.stride(0) == (hq + 2 * hkv) * d
    signs = _signs(d, 3)
    slots = torch.randperm(nb * 16, generator=g)[:T].to(torch.int64)
    slots[3] = -5           # padding
    slots[4] = nb * 16      # out of range -> skipped + status bit
    kc, vc, ks, vs = _empty(nb, hkv, d)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    qkv_d = qkv.cuda()
    _lib.write(qkv_d[:, hq * d:(hq + hkv) * d].view(T, hkv, d), qkv_d[:, (hq + hkv) * d:].view(T, hkv, d),
               slots.cuda(), kc, vc, ks, vs, signs.cuda(), dev_status=status)
    torch.cuda.synchronize()
    assert status.item() == _lib.DEV_BAD_SLOT
    ok = slots.clone()
    ok[4] = -1
    ref = _oracle_write(k.contiguous(), v.contiguous(), ok, nb, signs)
    got = [t.cpu().numpy() for t in (kc, vc, ks, vs)]
    for a, b in zip(got[2:], ref[2:]):
        assert np.array_equal(np.isnan(a), np.isnan(b))  # exactly the written slots changed
    written = np.zeros(nb * 16, bool)
    written[ok[ok >= 0].numpy()] = True
    written = written.reshape(nb, 16)
    assert np.array_equal(got[0][~written], ref[0][~written])
    diff = np.abs(O.unpack_codes(got[0][written]).astype(int) - O.unpack_codes(ref[0][written]).astype(int))
    assert diff.max() <= 1


def test_write_zero_tokens_and_bad_signs():
    d, hkv, nb = 96, 2, 4
    kc, vc, ks, vs = _empty(nb, hkv, d)
    before = kc.clone()
    empty = torch.zeros((0, hkv, d), dtype=torch.bfloat16, device="cuda")
    _lib.write(empty, empty, torch.zeros(0, dtype=torch.int64, device="cuda"), kc, vc, ks, vs,
               _signs(d, 1).cuda())
    torch.cuda.synchronize()
    assert torch.equal(kc, before)
    bad = _signs(d, 1)
    bad[5] = 0
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    x = torch.randn((3, hkv, d), device="cuda").to(torch.bfloat16)
    _lib.write(x, x, torch.arange(3, device="cuda"), kc, vc, ks, vs, bad.cuda(), dev_status=status)
    torch.cuda.synchronize()
    assert status.item() & _lib.DEV_BAD_SIGNS


def test_write_tiny_workload_matches_oracle_history():
    w = synthetic.make_workload("tiny")
    from int4_token_head_gb300.paged import PagedKV
    from tests.helpers import oracle_write_history_and_step
    pk = PagedKV(w)
    pk.populate_history(gen_device="cpu")
    q, k, v, slots = pk.step_inputs(gen_device="cpu")
    pk.write(k, v, slots)
    torch.cuda.synchronize()
    assert pk.status.item() == 0
    ref = oracle_write_history_and_step(w)
    got = [t.cpu().numpy() for t in (pk.k_cache, pk.v_cache, pk.k_scale, pk.v_scale)]
    # unused slots (the tail of seq 2's last block and the spare block) hold the sentinels
    assert np.array_equal(np.isnan(got[2]), np.isnan(ref[2]))
    mask = ~np.isnan(ref[2])
    diff = np.abs(O.unpack_codes(got[0][mask]).astype(int) - O.unpack_codes(ref[0][mask]).astype(int))
    assert diff.max() <= 1


@pytest.mark.parametrize("d,hkv", [(192, 40), (96, 36), (128, 70)])
def test_write_many_heads_generic_tiling(d, hkv):
    """More kv heads than fit whole tokens into one tile (the tile then spans
    token boundaries): codes and scales still bit-exact on the prerotated
    path, and within one code end to end."""
    T, nb = 53, 8
    ky = _rotated_inputs(T, hkv, d, 300 + d)
    vy = _rotated_inputs(T, hkv, d, 400 + d)
    g = torch.Generator().manual_seed(d + hkv)
    slots = torch.randperm(nb * 16, generator=g)[:T].to(torch.int64)
    got, status = _run_gpu_write(ky, vy, slots, nb, _signs(d, 0), prerotated=True)
    ref = _oracle_write(ky, vy, slots, nb, _signs(d, 0), prerotated=True)
    assert status == 0
    for a, b in zip(got, ref):
        if a.dtype == np.float32:
            assert np.array_equal(f32_bits(a), f32_bits(b))
        else:
            assert np.array_equal(a, b)
    k = torch.randn((T, hkv, d), generator=g).to(torch.bfloat16)
    got, status = _run_gpu_write(k, k, slots, nb, _signs(d, 5))
    ref = _oracle_write(k, k, slots, nb, _signs(d, 5))
    diff = np.abs(O.unpack_codes(got[0]).astype(int) - O.unpack_codes(ref[0]).astype(int))
    assert diff.max() <= 1
