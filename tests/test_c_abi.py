"""The boundary is a C ABI: both headers compile as strict C99 and a plain C program links
against the library and calls its host-only entry points (no GPU needed)."""

import ctypes
import os
import shutil
import subprocess

import pytest

from segmented_gather_gemm_lora_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stddef.h>
#include <stdio.h>
#include <string.h>
#include "lora_sgmv.h"
#include "lora_pool.h"

#define FIELD(T, f) printf(#T " " #f " %zu %zu\n", offsetof(T, f), sizeof(((T*)0)->f))

static void layouts(void) {
  printf("size lora_adapter_desc_t %zu\n", sizeof(lora_adapter_desc_t));
  FIELD(lora_adapter_desc_t, rank); FIELD(lora_adapter_desc_t, scale);
  FIELD(lora_adapter_desc_t, a_page0); FIELD(lora_adapter_desc_t, b_page0);
  printf("size lora_pool_view_t %zu\n", sizeof(lora_pool_view_t));
  FIELD(lora_pool_view_t, pool); FIELD(lora_pool_view_t, n_pages); FIELD(lora_pool_view_t, page_list);
  FIELD(lora_pool_view_t, n_page_list); FIELD(lora_pool_view_t, adapters); FIELD(lora_pool_view_t, n_adapters);
  FIELD(lora_pool_view_t, page_elems); FIELD(lora_pool_view_t, max_rank); FIELD(lora_pool_view_t, d_in);
  FIELD(lora_pool_view_t, d_out);
  printf("size lora_segments_t %zu\n", sizeof(lora_segments_t));
  FIELD(lora_segments_t, T); FIELD(lora_segments_t, max_long_units); FIELD(lora_segments_t, token_perm);
  FIELD(lora_segments_t, seg_indptr); FIELD(lora_segments_t, seg_adapter); FIELD(lora_segments_t, meta);
  FIELD(lora_segments_t, short_units); FIELD(lora_segments_t, long_units); FIELD(lora_segments_t, scratch);
  FIELD(lora_segments_t, h_scratch); FIELD(lora_segments_t, k_partials);
  printf("size lora_pool_stats_t %zu\n", sizeof(lora_pool_stats_t));
  FIELD(lora_pool_stats_t, hits); FIELD(lora_pool_stats_t, loads); FIELD(lora_pool_stats_t, refused);
  FIELD(lora_pool_stats_t, evictions); FIELD(lora_pool_stats_t, pages_loaded);
  FIELD(lora_pool_stats_t, resident); FIELD(lora_pool_stats_t, pinned);
}

int main(void) {
  lora_pool_stats_t st;
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
  if (lora_pool_mgr_stats(m, &st) != LORA_OK || st.loads != 2 || st.refused != 1 || st.evictions != 1 ||
      st.pages_loaded != 48 || st.resident != 0)
    return 13;
  lora_pool_mgr_destroy(m);
  layouts();
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
    lines = r.stdout.strip().splitlines()
    assert lines[-1] == "c abi ok"
    # the binding's ctypes structures lay out every field where the C compiler does
    structs = {"lora_adapter_desc_t": B.lora_adapter_desc_t, "lora_pool_view_t": B.lora_pool_view_t,
               "lora_segments_t": B.lora_segments_t, "lora_pool_stats_t": B.lora_pool_stats_t}
    seen = set()
    for line in lines[:-1]:
        parts = line.split()
        if parts[0] == "size":
            assert ctypes.sizeof(structs[parts[1]]) == int(parts[2]), line
            continue
        name, field, off, size = parts[0], parts[1], int(parts[2]), int(parts[3])
        desc = getattr(structs[name], field)
        assert (desc.offset, desc.size) == (off, size), line
        seen.add((name, field))
    for name, cls in structs.items():
        assert {f for f, _ in cls._fields_} == {f for n, f in seen if n == name}, name
