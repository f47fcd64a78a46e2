"""The boundary is a C ABI: both headers compile as strict C99 and a plain C program links
against the library and calls its host-only entry points (no GPU needed)."""

import os
import shutil
import subprocess

import pytest

from segmented_gather_gemm_lora_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "lora_sgmv.h"
#include "lora_pool.h"

int main(void) {
  lora_pool_mgr_t* m = NULL;
  int32_t pages[64], evicted[8], np = 0, ne = 0;
  if (lora_abi_version() != LORA_ABI_VERSION) return 1;
  if (strcmp(lora_status_string(LORA_OK), "ok") != 0) return 2;
  if (lora_pool_pages_needed(16, 4096, 4096, 4096) != 32) return 3;
  if (lora_segments_buffer_bytes(1000) == 0) return 4;
  if (lora_pool_mgr_create(40, 4096, 8, 16, 4096, 4096, &m) != LORA_OK || m == NULL) return 5;
  if (lora_pool_mgr_page_list_len(m) != 8 * 32) return 6;
  if (lora_pool_mgr_reserve(m, 3, 16, pages, 64, &np, evicted, 8, &ne) != LORA_OK || np != 32 || ne != 0) return 7;
  if (lora_pool_pin(m, 3) != LORA_OK) return 8;
  if (lora_pool_mgr_reserve(m, 4, 16, pages, 64, &np, evicted, 8, &ne) != LORA_ERR_WORKSPACE) return 9;
  if (lora_pool_unpin(m, 3) != LORA_OK) return 10;
  if (lora_pool_mgr_reserve(m, 4, 8, pages, 64, &np, evicted, 8, &ne) != LORA_OK || np != 16 || ne != 1 ||
      evicted[0] != 3 || lora_pool_resident_rank(m, 3) != 0)
    return 11;
  if (lora_pool_mgr_release(m, 4) != LORA_OK || lora_pool_mgr_free_pages(m) != 40) return 12;
  lora_pool_mgr_destroy(m);
  printf("c abi ok\n");
  return 0;
}
"""


def test_headers_compile_as_c99_and_a_c_program_links(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib = B.library_path()
    B.lib()  # built and loadable
    src = tmp_path / "abi.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "abi"
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
           str(src), "-o", str(exe), "-L", os.path.dirname(lib), "-l:" + os.path.basename(lib),
           "-Wl,-rpath," + os.path.dirname(lib)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stderr)
    assert r.stdout.strip() == "c abi ok"
