"""The C-ABI library builds, loads and exports every symbol include/kvint4.h
declares; host-side validation rejects bad arguments before any CUDA call.
No test here needs a GPU (no compute call is made)."""

import ctypes
import os
import re
import subprocess

import pytest

from int4_token_head_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvint4.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kv_int[48]_\w+)\s*\(", text)))


def _defines():
    text = open(HEADER).read()
    return {k: int(v) for k, v in re.findall(r"#define\s+(KV_INT4_\w+)\s+(\d+)", text)}


@pytest.fixture(scope="module")
def lib():
    return _lib.load()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert "kv_int4_write" in names and "kv_int4_attention" in names
    nm = subprocess.run(["nm", "-D", "--defined-only", build.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT\s+(\w+)", nm))
    for n in names:
        assert n in exported, n
        assert hasattr(lib, n)
    # nothing but the ABI is exported from our own code
    ours = {e for e in exported if e.startswith(("kv_int4", "kv_int8")) or "kvint4" in e}
    assert ours == set(names)


def test_binding_declares_every_symbol():
    assert set(_lib._SIGNATURES) == set(_declared())


def test_status_strings_and_version(lib):
    d = _defines()
    for name, code in d.items():
        if name.startswith("KV_INT4_ERR") or name == "KV_INT4_OK":
            s = lib.kv_int4_status_string(code).decode()
            assert s and s != "unknown status"
    assert lib.kv_int4_status_string(999).decode() == "unknown status"
    assert lib.kv_int4_version() == 4


def test_workspace_size_is_host_only_and_monotone(lib):
    a = lib.kv_int4_attention_workspace_size(256, 256, 32, 8, 128)
    b = lib.kv_int4_attention_workspace_size(512, 512, 32, 8, 128)
    assert 0 < a < b
    assert a % 256 == 0
    assert lib.kv_int4_attention_workspace_size(4, 4, 32, 7, 128) == 0   # heads not divisible
    assert lib.kv_int4_attention_workspace_size(4, 4, 32, 8, 100) == 0   # head size unsupported
    assert lib.kv_int4_attention_workspace_size(-1, 4, 32, 8, 128) == 0


D = _defines()
FAKE = ctypes.c_void_p(0x10000)       # never dereferenced: validation fails first
FAKE_ODD = ctypes.c_void_p(0x10008)   # 8-byte aligned only


def _write(lib, **kw):
    a = dict(k=FAKE, ks=8 * 128, v=FAKE, vs=8 * 128, slots=FAKE, nt=4, kc=FAKE, vc=FAKE, ksc=FAKE, vsc=FAKE,
             nb=4, bs=16, hkv=8, d=128, signs=FAKE, status=None, stream=None)
    a.update(kw)
    return lib.kv_int4_write(a["k"], a["ks"], a["v"], a["vs"], a["slots"], a["nt"], a["kc"], a["vc"], a["ksc"],
                             a["vsc"], a["nb"], a["bs"], a["hkv"], a["d"], a["signs"], a["status"], a["stream"])


def test_write_validation(lib):
    assert _write(lib, nt=0) == D["KV_INT4_OK"]
    assert _write(lib, k=None) == D["KV_INT4_ERR_NULL"]
    assert _write(lib, signs=None) == D["KV_INT4_ERR_NULL"]
    assert _write(lib, d=100) == D["KV_INT4_ERR_HEAD_SIZE"]
    assert _write(lib, d=80) == D["KV_INT4_ERR_HEAD_SIZE"]
    assert _write(lib, bs=32) == D["KV_INT4_ERR_BLOCK_SIZE"]
    assert _write(lib, hkv=0) == D["KV_INT4_ERR_HEADS"]
    assert _write(lib, nt=-1) == D["KV_INT4_ERR_SIZE"]
    assert _write(lib, k=FAKE_ODD) == D["KV_INT4_ERR_ALIGN"]
    assert _write(lib, kc=FAKE_ODD) == D["KV_INT4_ERR_ALIGN"]
    assert _write(lib, ks=8 * 128 + 4) == D["KV_INT4_ERR_ALIGN"]
    assert _write(lib, nt=1 << 28, hkv=8) == D["KV_INT4_ERR_SIZE"]
    assert _write(lib, slots=ctypes.c_void_p(0x10004)) == D["KV_INT4_ERR_ALIGN"]   # int64 slots: 8 bytes
    assert _write(lib, ksc=ctypes.c_void_p(0x10002)) == D["KV_INT4_ERR_ALIGN"]    # f32 scales: 4 bytes
    assert _write(lib, vsc=ctypes.c_void_p(0x10001)) == D["KV_INT4_ERR_ALIGN"]
    # the prerotated variant takes no signs
    r = lib.kv_int4_write_prerotated(FAKE, 1024, FAKE, 1024, FAKE, 0, FAKE, FAKE, FAKE, FAKE, 4, 16, 8, 128,
                                     None, None)
    assert r == D["KV_INT4_OK"]
    r = lib.kv_int4_write_prerotated(None, 1024, FAKE, 1024, FAKE, 3, FAKE, FAKE, FAKE, FAKE, 4, 16, 8, 128,
                                     None, None)
    assert r == D["KV_INT4_ERR_NULL"]


def _attn(lib, **kw):
    ws = lib.kv_int4_attention_workspace_size(2, 8, 32, 8, 128)
    a = dict(q=FAKE, qs=32 * 128, kc=FAKE, vc=FAKE, ksc=FAKE, vsc=FAKE, bt=FAKE, maxb=8, sl=FAKE, qsl=FAKE,
             ns=2, nq=8, mq=4, ms=128, hq=32, hkv=8, d=128, bs=16, nb=16, scale=0.1, causal=1, win=0, signs=FAKE,
             out=FAKE, os=32 * 128, ws=FAKE, wsb=ws, status=None, stream=None)
    a.update(kw)
    return lib.kv_int4_attention(a["q"], a["qs"], a["kc"], a["vc"], a["ksc"], a["vsc"], a["bt"], a["maxb"],
                                 a["sl"], a["qsl"], a["ns"], a["nq"], a["mq"], a["ms"], a["hq"], a["hkv"],
                                 a["d"], a["bs"], a["nb"], a["scale"], a["causal"], a["win"], a["signs"], a["out"],
                                 a["os"], a["ws"], a["wsb"], a["status"], a["stream"])


def test_attention_validation(lib):
    assert _attn(lib, ns=0) == D["KV_INT4_OK"]
    assert _attn(lib, nq=0) == D["KV_INT4_OK"]
    assert _attn(lib, q=None) == D["KV_INT4_ERR_NULL"]
    assert _attn(lib, signs=None) == D["KV_INT4_ERR_NULL"]
    assert _attn(lib, ws=None) == D["KV_INT4_ERR_WORKSPACE"]
    assert _attn(lib, wsb=1024) == D["KV_INT4_ERR_WORKSPACE"]
    assert _attn(lib, hkv=6) == D["KV_INT4_ERR_HEADS"]
    assert _attn(lib, hq=0) == D["KV_INT4_ERR_HEADS"]
    assert _attn(lib, hq=64 * 8) != D["KV_INT4_ERR_HEADS"] and _attn(lib, hq=65 * 8) == D["KV_INT4_ERR_HEADS"]
    assert _attn(lib, d=72) == D["KV_INT4_ERR_HEAD_SIZE"]
    assert _attn(lib, bs=8) == D["KV_INT4_ERR_BLOCK_SIZE"]
    assert _attn(lib, out=FAKE_ODD) == D["KV_INT4_ERR_ALIGN"]
    assert _attn(lib, ws=ctypes.c_void_p(0x10010)) == D["KV_INT4_ERR_ALIGN"]
    assert _attn(lib, qs=32 * 128 + 2) == D["KV_INT4_ERR_ALIGN"]
    for arg in ("ksc", "vsc", "bt", "sl", "qsl", "status"):
        assert _attn(lib, **{arg: ctypes.c_void_p(0x10002)}) == D["KV_INT4_ERR_ALIGN"], arg
    assert _attn(lib, ns=-3) == D["KV_INT4_ERR_SIZE"]
    assert _attn(lib, win=-1) == D["KV_INT4_ERR_SIZE"]
    assert _attn(lib, ns=0, win=4096) == D["KV_INT4_OK"]


def test_rht_validation(lib):
    def rht(x=FAKE, xs=128, y=FAKE, ys=128, f32=0, rows=4, d=128, signs=FAKE, inv=0):
        return lib.kv_int4_rht(x, xs, y, ys, f32, rows, d, signs, inv, None)
    assert rht(rows=0) == D["KV_INT4_OK"]              # nothing to do, nothing touched
    assert rht(rows=0, x=None, y=None, signs=None) == D["KV_INT4_OK"]
    assert rht(rows=-1) == D["KV_INT4_ERR_SIZE"]
    assert rht(d=0) == D["KV_INT4_ERR_HEAD_SIZE"]
    assert rht(d=4097) == D["KV_INT4_ERR_HEAD_SIZE"]
    assert rht(x=None) == D["KV_INT4_ERR_NULL"]
    assert rht(y=None) == D["KV_INT4_ERR_NULL"]
    assert rht(signs=None) == D["KV_INT4_ERR_NULL"]
    assert rht(x=ctypes.c_void_p(0x10001)) == D["KV_INT4_ERR_ALIGN"]
    assert rht(y=ctypes.c_void_p(0x10002), f32=1) == D["KV_INT4_ERR_ALIGN"]
    assert rht(xs=127) == D["KV_INT4_ERR_ALIGN"]
    assert rht(ys=100) == D["KV_INT4_ERR_ALIGN"]


def test_int8_entry_points_validation(lib):
    w = lambda **kw: lib.kv_int8_write(
        kw.get("k", FAKE), 8 * 128, FAKE, 8 * 128, FAKE, kw.get("nt", 4), kw.get("kc", FAKE), FAKE, FAKE, FAKE, 4,
        kw.get("bs", 16), 8, kw.get("d", 128), None, None)
    assert w(nt=0) == D["KV_INT4_OK"]
    assert w(k=None) == D["KV_INT4_ERR_NULL"]
    assert w(d=100) == D["KV_INT4_ERR_HEAD_SIZE"]
    assert w(bs=8) == D["KV_INT4_ERR_BLOCK_SIZE"]
    assert w(kc=FAKE_ODD) == D["KV_INT4_ERR_ALIGN"]
    ws = lib.kv_int4_attention_workspace_size(2, 8, 32, 8, 128)

    def a(**kw):
        return lib.kv_int8_attention(FAKE, 32 * 128, kw.get("kc", FAKE), FAKE, FAKE, FAKE, FAKE, 8, FAKE, FAKE,
                                     kw.get("ns", 2), 8, 4, 128, 32, 8, 128, 16, 16, 0.1, 1, kw.get("win", 0),
                                     kw.get("out", FAKE), 32 * 128, FAKE, ws, None, None)
    assert a(ns=0) == D["KV_INT4_OK"]
    assert a(out=None) == D["KV_INT4_ERR_NULL"]
    assert a(kc=FAKE_ODD) == D["KV_INT4_ERR_ALIGN"]
    assert a(win=-2) == D["KV_INT4_ERR_SIZE"]


def test_inslot_entry_points_validation(lib):
    assert lib.kv_int4_inslot_slot_bytes(128, 0) == 80
    assert lib.kv_int4_inslot_slot_bytes(96, 0) == 64
    assert lib.kv_int4_inslot_slot_bytes(128, 1) == 144
    assert lib.kv_int4_inslot_slot_bytes(100, 0) == 0
    w = lambda **kw: lib.kv_int4_write_inslot(FAKE, 8 * 128, FAKE, 8 * 128, FAKE, kw.get("nt", 4),
                                              kw.get("kv", FAKE), 4, 16, 8, kw.get("d", 128), kw.get("signs", FAKE),
                                              None, None)
    assert w(nt=0, kv=None) == D["KV_INT4_OK"]
    assert w(kv=None) == D["KV_INT4_ERR_NULL"]
    assert w(signs=None) == D["KV_INT4_ERR_NULL"]
    assert w(kv=FAKE_ODD) == D["KV_INT4_ERR_ALIGN"]
    assert w(d=72) == D["KV_INT4_ERR_HEAD_SIZE"]
    assert lib.kv_int8_write_inslot(FAKE, 1024, FAKE, 1024, FAKE, 4, None, 4, 16, 8, 128, None, None) == \
        D["KV_INT4_ERR_NULL"]
    ws = lib.kv_int4_attention_workspace_size(2, 8, 32, 8, 128)
    a = lambda **kw: lib.kv_int4_attention_inslot(FAKE, 32 * 128, kw.get("kv", FAKE), FAKE, 8, FAKE, FAKE,
                                                  kw.get("ns", 2), 8, 4, 128, 32, 8, 128, 16, 16, 0.1, 1, 0,
                                                  kw.get("signs", FAKE), FAKE, 32 * 128, FAKE, ws, None, None)
    assert a(ns=0) == D["KV_INT4_OK"]
    assert a(kv=None) == D["KV_INT4_ERR_NULL"]
    assert a(signs=None) == D["KV_INT4_ERR_NULL"]
    assert a(kv=FAKE_ODD) == D["KV_INT4_ERR_ALIGN"]


def test_selftest_wait_validation(lib):
    assert lib.kv_int4_selftest_wait(-1, FAKE, None, None) == D["KV_INT4_ERR_SIZE"]
    assert lib.kv_int4_selftest_wait(16, None, None, None) == D["KV_INT4_ERR_NULL"]
