"""The C ABI from C: a small C11 program compiled against include/topk_ragged.h
with -Wall -Wextra -Werror and linked to the built library calls every entry
point on its host-side paths (argument checks that fail before any device
work), so it needs no GPU.  This checks that the header is plain C and that
the library's symbols and return codes are what the header says."""
import os
import subprocess

import pytest

import sparse_attention_deterministic_gb300 as pkg
from sparse_attention_deterministic_gb300 import _native

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "topk_ragged.h"

#define CHECK(cond) do { if (!(cond)) { printf("FAIL %s\n", #cond); return 1; } } while (0)

int main(void)
{
    float *scores = (float *)0x1000;
    const int32_t *starts = (const int32_t *)0x2000, *lengths = (const int32_t *)0x3000;
    int32_t *out = (int32_t *)0x4000;
    CHECK(topk_ragged_abi_version() == TOPK_RAGGED_ABI_VERSION);
    CHECK(strcmp(topk_ragged_strerror(TOPK_OK), "ok") == 0);
    for (int s = TOPK_OK; s <= TOPK_ERR_CUDA; ++s) CHECK(topk_ragged_strerror(s) != NULL);
    /* argument checks fail before any device work */
    CHECK(topk_ragged(scores, 16, starts, lengths, 1, 0, TOPK_OFFSET_ROW_LOCAL, out, NULL, NULL)
          == TOPK_ERR_INVALID_ARG);
    CHECK(topk_ragged(scores, 16, starts, lengths, 1, TOPK_RAGGED_MAX_K + 1, 0, out, NULL, NULL)
          == TOPK_ERR_INVALID_ARG);
    CHECK(topk_ragged(scores, 16, starts, lengths, 1, 8, 4, out, NULL, NULL) == TOPK_ERR_INVALID_ARG);
    CHECK(topk_ragged(NULL, 0, NULL, NULL, 0, 8, TOPK_EXCLUDE_NEG_INF, NULL, NULL, NULL) == TOPK_OK);
    CHECK(topk_ragged_paged(scores, 16, starts, lengths, 1, 8, TOPK_OFFSET_ROW_START,
                            (const int32_t *)0x5000, 4, 64, out, NULL, NULL) == TOPK_ERR_INVALID_ARG);
    CHECK(topk_ragged_paged(scores, 16, starts, lengths, 1, 8, 0, (const int32_t *)0x5000, 4, 0, out, NULL,
                            NULL) == TOPK_ERR_INVALID_ARG);
    topk_row_stats *st = (topk_row_stats *)0x6000;
    CHECK(sizeof(topk_row_stats) == 6 * sizeof(uint32_t));
    CHECK(topk_ragged_stats(scores, 16, starts, lengths, 1, 0, st, NULL) == TOPK_ERR_INVALID_ARG);
    CHECK(topk_ragged_stats(NULL, 0, NULL, NULL, 0, 8, NULL, NULL) == TOPK_OK);
    CHECK(topk_ragged_indexer_scores((const uint16_t *)0x10000, (const float *)0x20000, NULL,
                                     (const uint16_t *)0x30000, 0, starts, lengths, starts, 1, 0.088f,
                                     scores, 16, NULL) == TOPK_ERR_INVALID_ARG);
    CHECK(topk_ragged_indexer((const uint16_t *)0x10000, (const float *)0x20000, NULL,
                              (const uint16_t *)0x30000, 100, starts, lengths, starts, 1, 0.088f, scores, 16,
                              8, TOPK_OFFSET_ROW_START, out, NULL, NULL) == TOPK_ERR_INVALID_ARG);
    CHECK(topk_ragged_device_status(NULL, NULL) == TOPK_ERR_INVALID_ARG);
    CHECK(topk_ragged_launch_info(16, 1, 8, NULL) == TOPK_ERR_INVALID_ARG);
    CHECK(TOPK_STAT_HAS_BOUNDARY == 1u && TOPK_STAT_STRADDLE == 2u && TOPK_STAT_ZERO_BOUND == 4u);
    CHECK(TOPK_DEV_LEN_ENVELOPE == 1u && TOPK_DEV_BAD_WINDOW == 2u && TOPK_DEV_INTERNAL == 4u);
    printf("OK\n");
    return 0;
}
"""


def test_header_is_c11_and_host_paths_answer_as_documented(tmp_path):
    pkg.build()
    lib_dir = os.path.dirname(_native.LIB_PATH)
    src = tmp_path / "abi.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "abi"
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
           "-o", str(exe), "-L", lib_dir, "-l:" + os.path.basename(_native.LIB_PATH), f"-Wl,-rpath,{lib_dir}"]
    build = subprocess.run(cmd, capture_output=True, text=True)
    if build.returncode != 0 and "cannot find" in build.stderr:
        pytest.skip(f"the library's runtime dependencies are not linkable here: {build.stderr.strip()[:200]}")
    assert build.returncode == 0, build.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0 and run.stdout.strip() == "OK", run.stdout + run.stderr
