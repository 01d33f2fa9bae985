"""include/attn.h is plain C: a C99 program compiles against it, links libattn.so and calls the
host-only entry points (no GPU needed)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_SOURCE = r"""
#include <stdio.h>
#include <string.h>
#include "attn.h"

int main(void) {
  if (attn_version() < 100) return 1;
  if (strcmp(attn_status_string(ATTN_ERR_WORKSPACE), "ATTN_ERR_WORKSPACE") != 0) return 2;
  /* the page's FA2 split counts: 431 blocks, four KV heads, capacity = 2 x SMs */
  if (attn_split_heuristic(4, 2 * 132, 431, 128) != 54) return 3;
  if (attn_split_heuristic(4, 2 * 148, 431, 128) != 62) return 4;
  if (attn_split_heuristic(4, 2 * 188, 431, 128) != 87) return 5;
  if (attn_decode_num_slots(480, 16, 0, 4096) != 2) return 6;
  if (attn_decode_workspace_bytes(2, 8, 128, 4) != (size_t)2 * 8 * 4 * 130 * 4) return 7;
  /* host argument checks return before any CUDA call */
  if (attn_prefill(NULL, NULL, NULL, NULL, NULL, 1, 1, 1, 1, 128, 0.1f, 1, NULL) != ATTN_ERR_INVALID_ARG) return 8;
  /* other backends' group counts at 27,525 tokens, four KV heads: XQA 33 on 132 SMs, 47 on 188 */
  if (attn_emulated_partitions(ATTN_NUMERICS_XQA, 1, 4, 27525, 132) != 33) return 9;
  if (attn_emulated_partitions(ATTN_NUMERICS_XQA, 1, 4, 27525, 188) != 47) return 10;
  if (attn_emulated_partitions(ATTN_NUMERICS_FA2, 1, 4, 27525, 148) != 62) return 11;
  if (attn_emulated_partitions(ATTN_NUMERICS_TRITON, 1, 4, 27525, 148) != 16) return 12;
  if (attn_emulated_num_slots(ATTN_NUMERICS_TRT, 1721, 16, 0) != 216) return 13;
  if (attn_emulated_workspace_bytes(2, 8, 128, 3) != (size_t)2 * 8 * 3 * 130 * 4) return 14;
  if (attn_merge_emulated(ATTN_NUMERICS_TRT, NULL, NULL, NULL, 1, 1, 128, NULL, NULL, NULL, NULL) !=
      ATTN_ERR_INVALID_ARG) return 15;
  puts("ok");
  return 0;
}
"""


def test_header_is_c_and_library_links(attn, tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "consumer.c"
    src.write_text(C_SOURCE)
    exe = tmp_path / "consumer"
    libdir = os.path.dirname(attn.library_path())
    subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                    "-L", libdir, "-lattn", f"-Wl,-rpath,{libdir}"], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.strip() == "ok", (out.returncode, out.stdout, out.stderr)
