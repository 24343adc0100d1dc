"""The boundary is a plain C ABI: a C99 program compiles against
include/rz.h with strict warnings, links librz.so and calls it (host-only
functions, and an entry point whose argument check fails before any CUDA
work).  CPU only."""

import os
import shutil
import subprocess

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <stdint.h>
#include "rz.h"

int main(void) {
  size_t ws = rz_workspace_size(RZ_OP_TOKEN_LOGPROB, 1000, 2560, 151936, 0);
  printf("ws %zu\n", ws);
  printf("text %s\n", rz_status_string(RZ_ERR_WORKSPACE));
  printf("scratch %zu\n", rz_noalloc_scratch_bytes());
  /* no workspace: refused by the argument check, nothing touches CUDA */
  int st = rz_token_logprob((const rz_bf16*)16, (const rz_bf16*)16, (const int32_t*)16, 5, 16,
                            100, (float*)16, NULL, NULL, 0, NULL, NULL);
  printf("call %d\n", st);
  return 0;
}
"""


def test_c_program_builds_links_and_calls(tmp_path):
    if torch.cuda.is_available():
        pytest.skip("fake-pointer calls are kept off machines with a GPU")
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    from invariant_logprobs_gb300 import build
    lib = build.build()
    src = tmp_path / "consumer.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "consumer"
    libdir = os.path.dirname(lib)
    cmd = [gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
           "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
           "-L", libdir, "-l:librz.so", "-Wl,-rpath," + libdir]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    lines = dict(l.split(" ", 1) for l in out.stdout.strip().splitlines())
    import invariant_logprobs_gb300 as rz
    assert int(lines["ws"]) == rz.workspace_size(rz.RZ_OP_TOKEN_LOGPROB, 1000, 2560, 151936, 0)
    assert lines["text"] == rz.status_string(rz.RZ_ERR_WORKSPACE)
    assert int(lines["scratch"]) == rz.noalloc_scratch_bytes()
    assert int(lines["call"]) == rz.RZ_ERR_WORKSPACE
