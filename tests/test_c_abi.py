"""The boundary is a plain C ABI: a C program (no C++, no Python, no torch)
includes include/nomas.h, links libnomas.so and calls its host-only entry
points.  Runs on the CPU; nothing here launches a kernel."""
import os
import shutil
import subprocess

import pytest

import segment_causal_kv_int8_b300 as nomas

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA_INC = "/usr/local/cuda/include"

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "nomas.h"

int main(void) {
  nomas_kvcache c;
  memset(&c, 0, sizeof(c));
  c.num_blocks = 54; c.heads = 16; c.head_dim = 128; c.grid_h = 23; c.grid_w = 40;
  c.capacity_frames = 18; c.past_frames = 18; c.dtype = NOMAS_INT8;
  c.k = (void*)256; c.v = (void*)512; c.k_scale = (float*)1024; c.v_scale = (float*)2048;
  if (nomas_kvcache_validate(&c) != NOMAS_OK) return 1;
  int32_t first = -1, slot = -1, valid = -1;
  int64_t total = -1;
  /* a 30-frame segment into an empty 18-frame window: its last 18 frames are written */
  if (nomas_kvcache_plan_append(&c, 30, &first, &slot, &total, &valid) != NOMAS_OK) return 2;
  printf("%d %s %zu %zu %d %d %lld %d\n", nomas_version(), nomas_status_string(NOMAS_ERR_CAPACITY),
         nomas_kvcache_bytes(&c), nomas_kvcache_archive_frame_bytes(&c), first, slot, (long long)total, valid);
  c.head_dim = 64;
  return nomas_kvcache_validate(&c) == NOMAS_ERR_UNSUPPORTED ? 0 : 3;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None or not os.path.exists(os.path.join(CUDA_INC, "cuda_runtime_api.h")),
                    reason="needs gcc and the CUDA headers")
def test_c_program_links_and_calls_the_library(tmp_path):
    src = tmp_path / "abi.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "abi"
    lib_dir = os.path.dirname(nomas.LIB_PATH)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), "-I", CUDA_INC,
                    str(src), "-o", str(exe), "-L", lib_dir, "-l:" + os.path.basename(nomas.LIB_PATH),
                    "-Wl,-rpath," + lib_dir], check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    assert int(out[0]) == nomas.nomas_version()
    slots = 54 * 16 * 18 * 920
    assert int(out[2]) == 2 * slots * (128 + 4)
    assert int(out[3]) == 2 * 54 * 16 * 920 * (128 + 4)
    # frames 12..29 are written; absolute frame 12 lives in ring slot 12 mod 18
    assert [int(x) for x in out[4:]] == [12, 12, 30, 18]
