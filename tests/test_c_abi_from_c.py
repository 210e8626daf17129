"""The public header is plain C: a C99 program includes it, links against
libfp8mla.so and calls the host-only entry points (no GPU needed)."""

import os
import shutil
import subprocess

import pytest

import paged_decode_attention_fp8_gb300 as fm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "fp8mla.h"

int main(void) {
  /* host-only calls: sizes, unit counts, status strings, refusals before any launch */
  if (fp8mla_metadata_units(152) != 76) return 1;
  if (fp8mla_workspace_bytes(64, 2, 64, 76) == 0) return 2;
  if (strcmp(fp8mla_status_string(FP8MLA_OK), "ok") != 0) return 3;
  if (paged_gqa_num_splits(1, 8, 16384, 152, 4) != 4) return 4;
  /* a foreign encoding is refused before anything touches the device */
  if (fp8mla_decode(NULL, NULL, FP8MLA_KV_E5M2, 1, NULL, 1, NULL, NULL, 0.04f, 1, NULL, NULL, 76, NULL, 0,
                    NULL, NULL, FP8MLA_DOT_FP8, 1, 2, 64, NULL) != FP8MLA_ERR_UNSUPPORTED_DTYPE) return 5;
  /* an empty cache write is accepted without a device */
  if (fp8_paged_cache_write(NULL, 128, NULL, 0, 1, 128, 16, 1, FP8MLA_KV_E4M3, NULL, NULL, (float*)8,
                            NULL) != FP8MLA_OK) return 6;
  printf("c abi ok\n");
  return 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
def test_header_compiles_as_c99_and_links(tmp_path):
    src = tmp_path / "abi.c"
    exe = tmp_path / "abi"
    src.write_text(PROGRAM)
    lib_dir = os.path.dirname(fm.LIB_PATH)
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I",
                        os.path.join(ROOT, "include"), str(src), "-o", str(exe), "-L", lib_dir, "-lfp8mla",
                        f"-Wl,-rpath,{lib_dir}"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stderr)
    assert r.stdout.strip() == "c abi ok"
