"""The launch planner on the CPU (no GPU needed): csrc/plan.h is plain host
arithmetic, so a small C++ program built against it checks, for every
k = 1..4096 and batches that reach every kernel variant on two device
shapes, that each CTA's shared-memory layout is aligned and fits its
variant's budget.  The staged keys are read and written as 16-byte vectors
and by 16-byte bulk copies, so their offset must stay a multiple of 16 bytes
(128 is kept) for every size of the candidate list before them, one 8-byte
slot at k <= 2 included."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "sparse_attention_deterministic_gb300", "csrc")

DRIVER = r"""
#include <stdio.h>
#include "plan.h"
using namespace topk_plan;

static int bad = 0;
#define CHECK(c) do { if (!(c)) { if (bad < 40) printf("k=%d B=%d n=%lld v=%d: %s\n", k, B, (long long)n, pl.variant, #c); ++bad; } } while (0)

static void shape(DeviceShape &d, int sms, int max_smem, int per_sm)
{
    d.sm_count = sms;
    d.max_smem = max_smem;
    d.smem_per_sm = per_sm;
    for (int c = 1; c <= 16; c *= 2) {
        d.max_clusters[kRowKernel][c] = 0;
        d.max_clusters[kCluster1024][c] = c == 16 ? sms / 19 : sms / c;     // GPC-bound at 16
        d.max_clusters[kCluster512][c] = c == 16 ? 2 * sms / 19 : 2 * sms / c;
    }
}

int main()
{
    DeviceShape devs[2];
    shape(devs[0], 152, 232448, 233472);   // GB300: 227 KB per block, 228 KB per SM
    shape(devs[1], 100, 101376, 102400);   // a smaller part: 99 KB per block
    const int Bs[] = {1, 2, 3, 4, 7, 16, 33, 64, 100, 128, 151, 152, 153, 200, 300, 400, 512, 607, 608, 1000, 16384};
    long long plans = 0;
    int seen[kVariants] = {0, 0, 0};
    for (const DeviceShape &dev : devs) {
        for (int k = 1; k <= 4096; ++k) {
            for (int B : Bs) {
                const long long ns[] = {(long long)B * 4096, (long long)B * 65536, (long long)B * 1048576, 2147483647LL};
                for (long long n : ns) {
                    if (n >= 2147483648LL || n < 0) continue;
                    const Plan pl = make_plan(n, B, k, dev);
                    ++plans;
                    seen[pl.variant] = 1;
                    const bool cl = pl.variant != kRowKernel;
                    CHECK(pl.off_win >= header_bytes(cl));
                    CHECK(pl.off_win % 16 == 0);
                    CHECK(pl.win_cap >= (cl ? (2 * k > 2048 ? 2 * k : 2048) : k - 1));
                    CHECK((pl.win_cap & (pl.win_cap - 1)) == 0);
                    CHECK(pl.off_keys % 128 == 0);
                    CHECK(pl.off_keys >= pl.off_win + 8 * pl.win_cap);
                    CHECK(pl.stage_cap % 128 == 0 && pl.stage_cap > 0);
                    CHECK(pl.stage_cap >= 2 * pl.win_cap);
                    CHECK(pl.smem == pl.off_keys + 4 * pl.stage_cap);
                    CHECK(4 * pl.stage_cap <= 8 * 32768);   // at most eight 32 KB copies per slice
                    CHECK(pl.smem <= dev.max_smem);
                    if (cl) {
                        CHECK(pl.smem <= variant_budget(dev, pl.variant));
                        CHECK(pl.cluster >= 2 && pl.cluster <= 16);
                        CHECK(pl.grid % pl.cluster == 0);
                        CHECK(pl.grid >= B);
                        CHECK(pl.grid / pl.cluster <= dev.max_clusters[pl.variant][pl.cluster]);
                        CHECK(B < 4 * dev.sm_count);
                    } else {
                        CHECK(pl.cluster == 1 && pl.grid == B);
                        CHECK(pl.stage_cap >= kShortScores);
                    }
                }
            }
        }
    }
    printf("plans %lld variants %d%d%d bad %d\n", plans, seen[0], seen[1], seen[2], bad);
    return bad != 0;
}
"""


def test_plan_layouts_aligned_and_within_budget(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    src = tmp_path / "plan_check.cpp"
    src.write_text(DRIVER)
    exe = tmp_path / "plan_check"
    subprocess.run([cxx, "-std=c++17", "-O2", "-Wall", "-Werror", "-I" + CSRC, str(src), "-o", str(exe)],
                   check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout[-4000:]
    # Every variant is reached by some batch.
    assert "variants 111" in out.stdout, out.stdout
