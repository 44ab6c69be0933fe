"""The boundary is a C ABI: include/kvint4.h compiles on its own as C99 and
as C++17 (no CUDA header needed), a C program links against libkvint4.so
and gets the documented validation results back, and concurrent calls from
several host threads return the same results as one thread.  No test here
needs a GPU: every call made stops at host-side validation."""

import ctypes
import os
import shutil
import subprocess
import threading

import pytest

from int4_token_head_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")

C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "kvint4.h"

#define CHECK(cond) do { if (!(cond)) { printf("FAILED line %d: %s\n", __LINE__, #cond); return 1; } } while (0)

int main(void) {
    /* addresses that validation rejects before any of them is dereferenced */
    void* dev = (void*)(uintptr_t)0x10000;
    int8_t* signs = (int8_t*)dev;
    size_t ws;
    CHECK(kv_int4_version() == 4);
    CHECK(strcmp(kv_int4_status_string(KV_INT4_OK), "ok") == 0);
    CHECK(strcmp(kv_int4_status_string(12345), "unknown status") == 0);
    ws = kv_int4_attention_workspace_size(2, 8, 32, 8, 128);
    CHECK(ws > 0 && ws % 256 == 0);
    CHECK(kv_int4_attention_workspace_size(2, 8, 32, 7, 128) == 0);
    /* write: empty batch, unsupported block size, head size, NULL, alignment */
    CHECK(kv_int4_write(dev, 1024, dev, 1024, (const int64_t*)dev, 0, (uint8_t*)dev, (uint8_t*)dev,
                        (float*)dev, (float*)dev, 4, 16, 8, 128, signs, NULL, NULL) == KV_INT4_OK);
    CHECK(kv_int4_write(dev, 1024, dev, 1024, (const int64_t*)dev, 4, (uint8_t*)dev, (uint8_t*)dev,
                        (float*)dev, (float*)dev, 4, 32, 8, 128, signs, NULL, NULL) == KV_INT4_ERR_BLOCK_SIZE);
    CHECK(kv_int4_write(dev, 1024, dev, 1024, (const int64_t*)dev, 4, (uint8_t*)dev, (uint8_t*)dev,
                        (float*)dev, (float*)dev, 4, 16, 8, 100, signs, NULL, NULL) == KV_INT4_ERR_HEAD_SIZE);
    CHECK(kv_int4_write(NULL, 1024, dev, 1024, (const int64_t*)dev, 4, (uint8_t*)dev, (uint8_t*)dev,
                        (float*)dev, (float*)dev, 4, 16, 8, 128, signs, NULL, NULL) == KV_INT4_ERR_NULL);
    CHECK(kv_int4_write(dev, 1024, dev, 1024, (const int64_t*)((char*)dev + 4), 4, (uint8_t*)dev,
                        (uint8_t*)dev, (float*)dev, (float*)dev, 4, 16, 8, 128, signs, NULL, NULL)
          == KV_INT4_ERR_ALIGN);
    /* attention: workspace too small, heads not divisible */
    CHECK(kv_int4_attention(dev, 4096, (const uint8_t*)dev, (const uint8_t*)dev, (const float*)dev,
                            (const float*)dev, (const int32_t*)dev, 8, (const int32_t*)dev, (const int32_t*)dev,
                            2, 8, 4, 128, 32, 8, 128, 16, 16, 0.1f, 1, 0, signs, dev, 4096, dev, 1024, NULL, NULL)
          == KV_INT4_ERR_WORKSPACE);
    CHECK(kv_int4_attention(dev, 4096, (const uint8_t*)dev, (const uint8_t*)dev, (const float*)dev,
                            (const float*)dev, (const int32_t*)dev, 8, (const int32_t*)dev, (const int32_t*)dev,
                            2, 8, 4, 128, 32, 6, 128, 16, 16, 0.1f, 1, 0, signs, dev, 4096, dev, ws, NULL, NULL)
          == KV_INT4_ERR_HEADS);
    /* the no-allocation variant rejects a call beyond its static scratch */
    CHECK(kv_int4_attention_noalloc(dev, 4096, (const uint8_t*)dev, (const uint8_t*)dev, (const float*)dev,
                                    (const float*)dev, (const int32_t*)dev, 8, (const int32_t*)dev,
                                    (const int32_t*)dev, 1000000, 1000000, 1, 128, 32, 8, 128, 16, 16, 0.1f, 1, 0,
                                    signs, dev, 4096, NULL, NULL) == KV_INT4_ERR_SCRATCH_LIMIT);
    /* the standalone rotation and the self-test take their stream as void* */
    CHECK(kv_int4_rht(dev, 128, dev, 128, 0, -1, 128, signs, 0, NULL) == KV_INT4_ERR_SIZE);
    CHECK(kv_int4_selftest_wait(-1, (int32_t*)dev, NULL, NULL) == KV_INT4_ERR_SIZE);
    CHECK(kv_int4_selftest_wait(4, NULL, NULL, NULL) == KV_INT4_ERR_NULL);
    printf("c boundary ok\n");
    return 0;
}
"""


def _compiler(names):
    for n in names:
        p = shutil.which(n)
        if p:
            return p
    pytest.skip(f"no compiler among {names}")


@pytest.mark.parametrize("lang", ["c99", "c11", "c++17"])
def test_header_compiles_without_cuda_headers(tmp_path, lang):
    cxx = lang.startswith("c++")
    cc = _compiler(["g++", "c++"] if cxx else ["gcc", "cc"])
    src = tmp_path / ("only_header.cpp" if cxx else "only_header.c")
    src.write_text('#include "kvint4.h"\nint kvint4_header_probe(void) { return KV_INT4_OK; }\n')
    cmd = [cc, f"-std={lang}", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", INCLUDE, "-c", str(src),
           "-o", str(tmp_path / "only_header.o")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_c_program_links_and_gets_validation_results(tmp_path):
    path = _lib.load()._name
    libdir = os.path.dirname(os.path.abspath(path))
    cc = _compiler(["gcc", "cc"])
    src = tmp_path / "abi_probe.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "abi_probe"
    cmd = [cc, "-std=c99", "-Wall", "-Werror", "-I", INCLUDE, str(src), "-o", str(exe), os.path.abspath(path),
           f"-Wl,-rpath,{libdir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c boundary ok" in r.stdout


def test_concurrent_validation_from_host_threads():
    """Many host threads calling the entry points at once (ctypes releases the
    GIL during the call) get exactly the single-threaded results."""
    lib = _lib.load()
    fake = ctypes.c_void_p(0x10000)
    misaligned = ctypes.c_void_p(0x10004)
    ws = lib.kv_int4_attention_workspace_size(2, 8, 32, 8, 128)
    results = []
    errors = []

    def worker(i):
        try:
            for _ in range(2000):
                a = lib.kv_int4_write(fake, 1024, fake, 1024, misaligned if i % 2 else fake, 4, fake, fake, fake,
                                      fake, 4, 16 if i % 2 else 8, 8, 128, fake, None, None)
                b = lib.kv_int4_attention(fake, 4096, fake, fake, fake, fake, fake, 8, fake, fake, 2, 8, 4, 128, 32,
                                          8, 128, 16, 16, 0.1, 1, 0, fake, fake, 4096, fake, 64, None, None)
                c = lib.kv_int4_attention_workspace_size(2, 8, 32, 8, 128)
                results.append((i % 2, a, b, c))
        except Exception as e:  # pragma: no cover - reported below
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(8)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors
    expect = {0: (_lib_code("KV_INT4_ERR_BLOCK_SIZE"), _lib_code("KV_INT4_ERR_WORKSPACE"), ws),
              1: (_lib_code("KV_INT4_ERR_ALIGN"), _lib_code("KV_INT4_ERR_WORKSPACE"), ws)}
    assert len(results) == 8 * 2000
    for parity, a, b, c in results:
        assert (a, b, c) == expect[parity]


def _lib_code(name):
    import re
    text = open(os.path.join(INCLUDE, "kvint4.h")).read()
    return int(re.search(rf"#define\s+{name}\s+(\d+)", text).group(1))
