"""The C ABI from C: ``include/pagedkv.h`` compiles as C99 (gcc -std=c99
-Wall -Werror), a program links against ``libpagedkv.so`` and drives the host
block pool through it (no GPU call).  The program replays the nano-vLLM
section 4.2 sizing and a FIFO / slot trace that the oracle pool also gives."""
import os
import shutil
import subprocess

import numpy as np
import pytest

from oracle import pool as OP

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIB_DIR = os.path.join(ROOT, "paged_kv_cache_295_gb300")

C_SOURCE = r"""
#include <stdio.h>
#include "pagedkv.h"

#define CHECK(x) do { pkv_status s_ = (x); if (s_ != PKV_OK) { \
    fprintf(stderr, "%s -> %d\n", #x, (int)s_); return 1; } } while (0)

int main(void) {
  /* 4 blocks, freed in a shuffled initial order */
  const int32_t order[4] = {2, 0, 3, 1};
  pkv_pool_config cfg = {0};
  cfg.num_layers = 2; cfg.num_kv_heads = 2; cfg.head_dim = 64; cfg.block_size = 4;
  cfg.kv_dtype = PKV_BF16; cfg.num_blocks = 4; cfg.initial_free_order = order;
  printf("block_bytes %lld\n", (long long)pkv_block_bytes(&cfg));
  pkv_pool* pool = NULL;
  CHECK(kv_pool_init(&cfg, &pool));
  CHECK(seq_create(pool, 7));
  CHECK(seq_create(pool, 9));
  int64_t slots[6];
  CHECK(seq_append_tokens(pool, 7, 6, slots));
  for (int i = 0; i < 6; ++i) printf("slot %lld\n", (long long)slots[i]);
  int64_t ids[2] = {7, 9}, step[2];
  CHECK(seq_append_slots(pool, ids, 2, step));
  printf("step %lld %lld\n", (long long)step[0], (long long)step[1]);
  pkv_pool_stats st;
  CHECK(kv_pool_stats(pool, &st));
  printf("used %lld free %lld\n", (long long)st.used_blocks, (long long)st.free_blocks);
  int32_t blk = -1;
  pkv_status s = block_alloc(pool, &blk);
  printf("alloc %d %d\n", (int)s, (int)blk);
  s = block_alloc(pool, &blk);
  printf("alloc_empty %d\n", (int)(s == PKV_ERR_NO_FREE_BLOCK));
  CHECK(seq_free(pool, 7));
  CHECK(kv_pool_stats(pool, &st));
  printf("after_free %lld\n", (long long)st.free_blocks);
  kv_pool_destroy(pool);
  return 0;
}
"""


@pytest.fixture(scope="module")
def c_program(tmp_path_factory, lib):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    d = tmp_path_factory.mktemp("cabi")
    src = d / "main.c"
    src.write_text(C_SOURCE)
    exe = d / "main"
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I",
                    os.path.join(ROOT, "include"), str(src), "-o", str(exe), "-L", LIB_DIR,
                    "-lpagedkv", "-Wl,-rpath," + LIB_DIR], check=True)
    return exe


def test_header_is_c_and_the_pool_runs_from_c(c_program):
    out = subprocess.run([str(c_program)], check=True, capture_output=True, text=True).stdout
    lines = dict(l.split(" ", 1) for l in out.strip().splitlines() if not l.startswith("slot "))
    slots = [int(l.split()[1]) for l in out.splitlines() if l.startswith("slot ")]
    # 2 (K, V) x 2 layers x 4 tokens x 2 heads x 64 dims x 2 bytes
    assert int(lines["block_bytes"]) == 2 * 2 * 4 * 2 * 64 * 2
    op = OP.Pool(2, 2, 64, 4, 2, 4, initial_free_order=[2, 0, 3, 1])
    op.seq_create(7)
    op.seq_create(9)
    assert slots == op.seq_append_tokens(7, 6)
    assert [int(x) for x in lines["step"].split()] == op.seq_append_slots([7, 9])
    # sequence 7 holds 2 blocks (7 tokens), sequence 9 one: one block is left
    used, free = (int(x) for x in lines["used"].replace("free", "").split())
    assert (used, free) == (4 - len(op.free), len(op.free)) == (3, 1)
    status, blk = (int(x) for x in lines["alloc"].split())
    assert status == 0 and blk == list(op.free)[0]       # the free list's front
    assert lines["alloc_empty"] == "1"                   # then NO_FREE_BLOCK
    assert int(lines["after_free"]) == 2                 # sequence 7's two blocks came back
