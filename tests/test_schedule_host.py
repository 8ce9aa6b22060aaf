"""Host-side checks of the decode schedule's arithmetic (csrc/common.cuh).

The chunk order of a batch is cut into one contiguous range per worker
(range_begin / worker_of); the segment of unit u in worker w's range keeps its
partial state in slot u + w, and a split unit's merge reads the slots of the
workers from worker_of(first chunk) to worker_of(last chunk).  A small host
program built with nvcc from the library's own header checks, by brute force
over many chunk totals, worker counts and random unit layouts, that:

* the ranges tile [0, T) in order, the first T mod NW of them one chunk longer;
* worker_of(f) is the range holding f;
* the slots of all segments are distinct and below U + NW, and a unit that lies
  in one range has exactly one segment.

A second program checks RowShape, the map from a unit's rows to rows of q /
out when a sequence has several query tokens.
"""
from __future__ import annotations

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "paged_kv_decode_16_gb300", "csrc")
INCLUDE = os.path.join(ROOT, "include")

PROGRAM = r"""
#include <cstdio>
#include <cstdlib>
#include <vector>
#include "common.cuh"
using namespace pkv;

static unsigned long long rng = 88172645463325252ull;
static unsigned next_u32() {
    rng ^= rng << 13; rng ^= rng >> 7; rng ^= rng << 17;
    return (unsigned)(rng >> 11);
}

int main() {
    long long checks = 0;
    // ranges: tiling, lengths, inverse
    for (int T = 1; T <= 600; T += (T < 80 ? 1 : 13)) {
        for (int nw = 1; nw <= T && nw <= 300; nw += (nw < 24 ? 1 : 17)) {
            const int sw = T / nw, r = T % nw;
            if (range_begin(0, sw, r) != 0 || range_begin(nw, sw, r) != T) {
                printf("FAIL ends T=%d nw=%d\n", T, nw);
                return 1;
            }
            for (int w = 0; w < nw; ++w) {
                const int len = range_begin(w + 1, sw, r) - range_begin(w, sw, r);
                if (len != sw + (w < r ? 1 : 0)) {
                    printf("FAIL len T=%d nw=%d w=%d\n", T, nw, w);
                    return 1;
                }
                for (int f = range_begin(w, sw, r); f < range_begin(w + 1, sw, r); ++f)
                    if (worker_of(f, sw, r) != w) {
                        printf("FAIL worker_of T=%d nw=%d f=%d\n", T, nw, f);
                        return 1;
                    }
            }
            ++checks;
        }
    }
    // slots of random unit layouts
    for (int trial = 0; trial < 3000; ++trial) {
        const int U = 1 + next_u32() % 60;
        std::vector<int> nch(U);
        int T = 0;
        for (int u = 0; u < U; ++u) {
            const unsigned k = next_u32() % 10;
            nch[u] = k < 2 ? 0 : (k < 6 ? 1 + next_u32() % 8 : 1 + next_u32() % 400);
            T += nch[u];
        }
        if (T == 0) continue;
        const int nw = 1 + next_u32() % (T < 200 ? T : 200);
        const int sw = T / nw, r = T % nw;
        std::vector<int> used(U + nw, 0);
        int a = 0;
        for (int u = 0; u < U; ++u) {
            if (nch[u] == 0) continue;
            const int w0 = worker_of(a, sw, r), w1 = worker_of(a + nch[u] - 1, sw, r);
            const bool inside = range_begin(w0, sw, r) <= a &&
                                a + nch[u] <= range_begin(w0 + 1, sw, r);
            if (inside != (w0 == w1)) {
                printf("FAIL inside trial=%d u=%d\n", trial, u);
                return 1;
            }
            for (int w = w0; w <= w1; ++w) {
                const int slot = u + w;
                if (slot >= U + nw || used[slot]++) {
                    printf("FAIL slot trial=%d u=%d w=%d\n", trial, u, w);
                    return 1;
                }
            }
            a += nch[u];
        }
        ++checks;
    }
    printf("ok %lld\n", checks);
    return 0;
}
"""


def _nvcc():
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "bin", "nvcc")):
            return os.path.join(cand, "bin", "nvcc")
    return shutil.which("nvcc")


def test_schedule_ranges_and_slots(tmp_path):
    nvcc = _nvcc()
    if not nvcc:
        pytest.skip("nvcc is needed to build the host check against the CUDA header")
    src = tmp_path / "schedule_check.cu"
    exe = tmp_path / "schedule_check"
    src.write_text(PROGRAM)
    build = subprocess.run([nvcc, "-std=c++17", "-I", INCLUDE, "-I", CSRC, str(src), "-o",
                            str(exe)], capture_output=True, text=True)
    assert build.returncode == 0, build.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0 and run.stdout.startswith("ok"), run.stdout + run.stderr


ROWSHAPE_PROGRAM = r"""
#include <cstdio>
#include <vector>
#include "common.cuh"
using namespace pkv;

int main() {
    long long checks = 0;
    const int B = 3, Hkv = 2;
    for (int group = 1; group <= 12; ++group)
    for (int hpu = 1; hpu <= group; ++hpu) {
        if (group % hpu) continue;
        for (int qn = 1; qn <= 64; qn += (qn < 20 ? 1 : 7))
        for (int qpu = 1; qpu <= qn && qpu * hpu <= 32; ++qpu) {
            const int tiles = (qn + qpu - 1) / qpu;
            const int hq = group * Hkv;
            RowShape rs{qn, qpu, hpu, group / hpu, group, hq};
            const int sub_groups = rs.head_blocks * tiles;
            std::vector<int> hit((size_t)B * qn * hq, 0);
            for (int b = 0; b < B; ++b)
            for (int h = 0; h < Hkv; ++h)
            for (int sg = 0; sg < sub_groups; ++sg) {
                const int n = rs.rows(sg);
                if (n < 1 || n > qpu * hpu) { printf("FAIL rows\n"); return 1; }
                for (int r = 0; r < n; ++r) {
                    const long long row = rs.row(b, h, sg, r);
                    if (row < 0 || row >= (long long)B * qn * hq) { printf("FAIL range\n"); return 1; }
                    hit[row]++;
                    // the row's token is query(sg, r), its head belongs to KV head h
                    const long long j = (row / hq) % qn, head = row % hq;
                    if (j != rs.query(sg, r) || head / group != h || row / ((long long)qn * hq) != b) {
                        printf("FAIL token/head g=%d hpu=%d qn=%d qpu=%d\n", group, hpu, qn, qpu);
                        return 1;
                    }
                }
            }
            for (size_t i = 0; i < hit.size(); ++i)
                if (hit[i] != 1) {
                    printf("FAIL cover g=%d hpu=%d qn=%d qpu=%d row=%zu n=%d\n", group, hpu, qn, qpu, i, hit[i]);
                    return 1;
                }
            ++checks;
        }
    }
    printf("ok %lld\n", checks);
    return 0;
}
"""


def test_row_shape_covers_every_query_row_once(tmp_path):
    """RowShape (several query tokens per sequence): for every tile length,
    head block and query count, the rows of all units (b, KV head, sub-group)
    hit each row of q / out [B][Qn][Hq] exactly once, at the token query()
    names and a head of the unit's KV head."""
    nvcc = _nvcc()
    if not nvcc:
        pytest.skip("nvcc is needed to build the host check against the CUDA header")
    src = tmp_path / "rowshape_check.cu"
    exe = tmp_path / "rowshape_check"
    src.write_text(ROWSHAPE_PROGRAM)
    build = subprocess.run([nvcc, "-std=c++17", "-I", INCLUDE, "-I", CSRC, str(src), "-o",
                            str(exe)], capture_output=True, text=True)
    assert build.returncode == 0, build.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0 and run.stdout.startswith("ok"), run.stdout + run.stderr
