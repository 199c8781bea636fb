"""The C ABI from C: a C99 program includes include/pkv.h, links libpkv.so and calls the
host-validated paths (no GPU needed): status names, argument errors, struct layout."""
import os
import subprocess

import pytest

from paged_kv_attention_09_gb300 import pkv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <stddef.h>
#include <string.h>
#include "pkv.h"

int main(void) {
  pkv_cache c;
  memset(&c, 0, sizeof c);
  c.k_cache = (void*)0x10000; c.v_cache = (void*)0x20000;
  c.num_pages = 8; c.page_size = 16; c.num_kv_heads = 2; c.head_dim = 64;
  c.kv_dtype = PKV_BF16; c.window = 0;
  size_t n = 0;
  printf("sizeof %zu %zu %zu\n", sizeof(pkv_cache), offsetof(pkv_cache, window),
         sizeof(pkv_decode_graph_desc));
  printf("null %d\n", (int)pkv_append(NULL, 0, 0, PKV_F32, 0, 1, NULL, NULL));
  c.page_size = 8;
  printf("page %d\n", (int)pkv_append(&c, (void*)0x30000, (void*)0x40000, PKV_F32,
                                     (const int32_t*)0x50000, 1, NULL, NULL));
  c.page_size = 16; c.window = -1;
  printf("window %d\n", (int)pkv_decode_workspace_size(&c, 1, 4, 4, &n));
  c.window = 0; c.kv_dtype = 9;
  printf("dtype %d\n", (int)pkv_decode_workspace_size(&c, 1, 4, 4, &n));
  printf("graph %d\n", (int)pkv_decode_graph_launch(NULL, 1, NULL));
  printf("name %s\n", pkv_status_string(PKV_ERR_WORKSPACE));
  printf("formats %d %d %d %d %d\n", PKV_F32, PKV_BF16, PKV_INT8, PKV_FP8, PKV_INT4);
  return 0;
}
"""


def test_c_program_compiles_links_and_validates(tmp_path):
    if not os.path.exists(pkv.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    src = tmp_path / "abi.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "abi"
    libdir = os.path.dirname(pkv.LIB_PATH)
    cc = ["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
          str(src), "-o", str(exe), "-L", libdir, "-l:libpkv.so", f"-Wl,-rpath,{libdir}"]
    r = subprocess.run(cc, capture_output=True, text=True)
    if r.returncode != 0 and "cannot find" in r.stderr:
        pytest.skip("linker cannot find the library's CUDA runtime: " + r.stderr[-200:])
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    got = dict(line.split(" ", 1) for line in out.stdout.strip().splitlines())
    import ctypes
    sizes = [int(x) for x in got["sizeof"].split()]
    assert sizes[0] == ctypes.sizeof(pkv.pkv_cache)            # the binding's struct layout
    assert sizes[1] == pkv.pkv_cache.window.offset
    assert sizes[2] == ctypes.sizeof(pkv.pkv_decode_graph_desc)
    assert got["null"] == "1" and got["page"] == "4" and got["window"] == "2"
    assert got["dtype"] == "3" and got["graph"] == "1"
    assert got["name"].startswith("PKV_ERR_WORKSPACE")
    assert got["formats"] == "0 1 2 3 4"
