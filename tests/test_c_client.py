"""The boundary from plain C: include/fia.h compiles as C99 with every warning
on, and a C program linked against libfia.so validates shapes through it
(no CUDA call is made on these paths)."""
import os
import shutil
import subprocess

import pytest

from attention_fia_prefill_gb300 import build as fia_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_SRC = r"""
#include <stdio.h>
#include <string.h>
#include "fia.h"

static fia_tensor t4(int32_t dtype, int64_t a, int64_t b, int64_t c, int64_t d) {
  fia_tensor t;
  memset(&t, 0, sizeof t);
  t.data = (void*)(1 << 20);   /* never dereferenced: validation only */
  t.dtype = dtype;
  t.ndim = 4;
  t.shape[0] = a; t.shape[1] = b; t.shape[2] = c; t.shape[3] = d;
  return t;
}

int main(void) {
  fia_params p;
  size_t ws = 0;
  fia_tensor q = t4(FIA_DTYPE_BF16, 2, 4, 300, 128), k = t4(FIA_DTYPE_BF16, 2, 2, 300, 128);
  fia_tensor k64 = t4(FIA_DTYPE_BF16, 2, 2, 300, 64);
  fia_params_init(&p);
  p.num_heads = 4;
  p.num_key_value_heads = 2;
  p.input_layout = "BNSD";
  p.sparse_mode = 3;
  printf("%d\n", (int)fia_prefill_get_workspace_size(&q, &k, &k, NULL, &p, &q, NULL, &ws));
  printf("%d\n", ws > 0);
  printf("%d\n", (int)fia_prefill_get_workspace_size(&q, &k64, &k64, NULL, &p, &q, NULL, &ws));
  p.sparse_mode = 9;
  printf("%d\n", (int)fia_prefill_get_workspace_size(&q, &k, &k, NULL, &p, &q, NULL, &ws));
  printf("%s\n", fia_status_string(FIA_ERR_SPARSE_MODE));
  return 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_c99_client(tmp_path):
    lib = fia_build.build()
    src = tmp_path / "client.c"
    src.write_text(C_SRC)
    exe = tmp_path / "client"
    libdir = os.path.dirname(lib)
    cc = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I",
                         os.path.join(ROOT, "include"), str(src), "-L", libdir, "-lfia", f"-Wl,-rpath,{libdir}",
                         "-o", str(exe)], capture_output=True, text=True)
    assert cc.returncode == 0, cc.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0, run.stderr
    lines = run.stdout.split()
    assert lines[:4] == ["0", "1", "3", "12"], run.stdout
    assert "FIA_ERR_SPARSE_MODE" in run.stdout
