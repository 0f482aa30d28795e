"""The boundary from plain C: `include/kvq.h` compiles as C99 with warnings as
errors (no C++ or torch types leak into it), and a C program linked against
libkvq.so calls the host-only entry points and gets the documented status
codes for invalid arguments -- all before any CUDA call, so no GPU is needed."""
import os
import shutil
import subprocess

import pytest

import int8_quantized_paged_tokenwise_gb300 as kvq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OUT = os.path.join(ROOT, "int8_quantized_paged_tokenwise_gb300", "_build", "c_abi_check")

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "kvq.h"

int main(void) {
  int fails = 0;
  if (kvq_version() != 100) { puts("version"); ++fails; }
  if (strcmp(kvq_status_string(KVQ_OK), "ok") != 0) { puts("status string"); ++fails; }
  /* an unsupported block size, a NULL query, and the empty no-op */
  char buf[64];
  void* p = (void*)(((unsigned long)buf + 15) & ~15ul);
  kvq_status s = kvq_paged_decode(p, KVQ_BF16, 2, 8, 2, 128, (const int8_t*)p, (const int8_t*)p,
                                  (const uint16_t*)p, (const uint16_t*)p, 16, 32,
                                  (const int32_t*)p, 4, (const int32_t*)p, 64, 0.1f, p, NULL, 0,
                                  NULL);
  if (s != KVQ_ERR_UNSUPPORTED) { printf("block size: %d\n", (int)s); ++fails; }
  s = kvq_paged_decode(NULL, KVQ_BF16, 2, 8, 2, 128, (const int8_t*)p, (const int8_t*)p,
                       (const uint16_t*)p, (const uint16_t*)p, 16, 16, (const int32_t*)p, 4,
                       (const int32_t*)p, 64, 0.1f, p, NULL, 0, NULL);
  if (s != KVQ_ERR_INVALID_ARGUMENT) { printf("null q: %d\n", (int)s); ++fails; }
  s = kvq_quantize_append(p, p, 256, 256, 0, 2, 128, KVQ_FP16, (const int64_t*)p, (int8_t*)p,
                          (int8_t*)p, (uint16_t*)p, (uint16_t*)p, 16, 16, NULL);
  if (s != KVQ_OK) { printf("empty append: %d\n", (int)s); ++fails; }
  if (kvq_decode_workspace_bytes(0, 8, 2, 128, 64) != 0) { puts("workspace of B=0"); ++fails; }
  printf(fails ? "FAIL %d\n" : "ok\n", fails);
  return fails != 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_header_is_c99_and_the_library_links_from_c():
    lib = kvq.load()
    os.makedirs(OUT, exist_ok=True)
    src = os.path.join(OUT, "abi_check.c")
    exe = os.path.join(OUT, "abi_check")
    with open(src, "w") as f:
        f.write(PROGRAM)
    libdir = os.path.dirname(str(kvq.LIB_PATH))
    cc = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                         "-I", os.path.join(ROOT, "include"), src, "-o", exe,
                         "-L", libdir, "-lkvq", "-Wl,-rpath," + libdir],
                        capture_output=True, text=True)
    assert cc.returncode == 0, cc.stderr
    run = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0 and run.stdout.strip() == "ok", run.stdout + run.stderr
    assert lib is not None
