"""The C ABI from C: include/ll.h compiles as plain C11 and libll.so links and runs.

A small C program (no C++, no CUDA headers) includes the header, links the
library and calls the entry points that need no device: the status strings, the
launch counter, and the frame-to-slot map and resident list of "LongLive" §3.3
("Frame sink": the sink frames stay; the window rolls with FIFO eviction).  Its
output is checked against the float64 oracle's bookkeeping, and cache creation
without a device must fail cleanly (a status, a NULL handle).
"""

import os
import shutil
import subprocess

import pytest

import oracle
from tests.conftest import ROOT

PROGRAM = r"""
#include <stdio.h>
#include <stdint.h>
#include "ll.h"

int main(void) {
  int s, w;
  int64_t f, n, frames[64];
  printf("status %s|%s\n", ll_status_str(LL_OK), ll_status_str(LL_ERR_UNSUPPORTED));
  printf("launches %llu\n", (unsigned long long)ll_launch_count());
  for (s = 0; s <= 4; ++s)
    for (w = 0; w <= 5; ++w) {
      for (f = 0; f < 24; ++f) printf("slot %d %d %lld %d\n", s, w, (long long)f, ll_frame_slot(s, w, f));
      for (n = 0; n < 24; ++n) {
        int i, r = ll_resident_frames(s, w, n, frames);
        printf("res %d %d %lld", s, w, (long long)n);
        for (i = 0; i < r; ++i) printf(" %lld", (long long)frames[i]);
        printf("\n");
      }
    }
  {
    ll_cache* c = (ll_cache*)&s;  /* must come back NULL on failure */
    ll_status st = ll_cache_create(&c, 1, 2, 64, 16, 3, 6, 3, LL_BF16);
    printf("create %d %s\n", st == LL_OK ? 0 : 1, c == NULL ? "null" : "handle");
    if (st == LL_OK) ll_cache_destroy(c);
  }
  return 0;
}
"""


@pytest.fixture(scope="module")
def lib_path():
    from windowed_sink_attention_ll_b300 import build_lib

    build_lib.build()
    path = os.path.join(ROOT, "windowed_sink_attention_ll_b300", "libll.so")
    assert os.path.exists(path)
    return path


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs a C compiler")
def test_header_compiles_as_c_and_the_library_runs_from_c(lib_path, tmp_path):
    src = tmp_path / "abi.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "abi"
    libdir = os.path.dirname(lib_path)
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I" + os.path.join(ROOT, "include"),
           str(src), "-o", str(exe), lib_path, "-Wl,-rpath," + libdir]
    out = subprocess.run(cmd, capture_output=True, text=True)
    assert out.returncode == 0, out.stderr
    env = dict(os.environ)
    env.pop("CUDA_VISIBLE_DEVICES", None)
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120, env=env)
    assert run.returncode == 0, run.stderr
    lines = run.stdout.splitlines()
    assert lines[0] == "status LL_OK|LL_ERR_UNSUPPORTED"
    assert lines[1] == "launches 0"
    slots = res = 0
    for line in lines[2:]:
        tok = line.split()
        if tok[0] == "slot":
            S, W, f, got = map(int, tok[1:])
            want = oracle.slot_of_frame(S, W, f) if (f < S or W > 0) else -1
            assert got == want, line
            slots += 1
        elif tok[0] == "res":
            S, W, n = map(int, tok[1:4])
            assert [int(x) for x in tok[4:]] == oracle.resident_frames(S, W, n), line
            res += 1
    assert slots == res == 5 * 6 * 24
    create = [line for line in lines if line.startswith("create")]
    assert len(create) == 1
    if create[0] != "create 0 handle":  # no device here: a status and a NULL handle
        assert create[0] == "create 1 null", create[0]
