"""The record layout on the host (no GPU): the chunk record's offsets are
disjoint and in range, and p_chunk numbers the 16-byte chunks of P's lower
triangle (row r, 8-column chunk c <= r / 8) one to one onto 0 .. 287, rows in
order.  A small host program includes the layout header and prints what it
computes; nvcc compiles it (host code only).  The bench's byte accounting
carries its own copy of the record size, checked against the header here."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "gated_delta_rule_04_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include "kda_chunk_layout.cuh"
int main() {
    std::printf("%d %d %d %d %d %d %d %d\n", kda::REC_W, kda::REC_Q, kda::REC_PANEL, kda::REC_KT, kda::REC_UT,
                kda::REC_P, kda::REC_DECAY, kda::REC_BYTES);
    for (int r = 0; r < 64; ++r)
        for (int c = 0; c <= r / 8; ++c) std::printf("%d %d %d\n", r, c, kda::p_chunk(r, c));
    return 0;
}
"""


@pytest.fixture(scope="module")
def layout(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc is not available")
    d = tmp_path_factory.mktemp("layout")
    src, exe = d / "layout.cu", d / "layout"
    src.write_text(PROGRAM)
    subprocess.run([nvcc, "-std=c++17", "-I", os.path.join(ROOT, "include"), "-I", CSRC, str(src), "-o", str(exe)],
                   check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    offsets = [int(x) for x in out[0].split()]
    chunks = [tuple(int(x) for x in line.split()) for line in out[1:] if line.strip()]
    return offsets, chunks


def test_record_parts_are_disjoint_and_in_range(layout):
    (w, q, panel, kt, ut, p, decay, total), _ = layout
    # [W; Q+] panels: W and Q+ rows of keys 0-63, then of keys 64-127, 8 KiB each
    parts = [(w, 8192), (q, 8192), (w + panel, 8192), (q + panel, 8192),
             (kt, 128 * 64 * 2), (ut, 128 * 64 * 2), (p, 288 * 16), (decay, 128 * 4)]
    parts.sort()
    for (a, n), (b, _) in zip(parts, parts[1:]):
        assert a + n <= b, "record parts overlap"
    assert parts[0][0] == 0 and parts[-1][0] + parts[-1][1] == total
    # every tile an MMA reads straight from the record starts on 1 KiB
    for off in (w, q, w + panel, q + panel, kt, ut):
        assert off % 1024 == 0
    # two bulk copies of 16-byte multiples move a record
    assert total % 32 == 0


def test_p_chunk_numbers_the_lower_triangle_in_row_order(layout):
    _, chunks = layout
    assert len(chunks) == 288   # sum over 64 rows of (r / 8 + 1)
    indices = [i for _, _, i in chunks]
    assert indices == list(range(288)), "p_chunk is not the row-major enumeration of the triangle"
    # the chunks past r / 8 are the ones every element of which lies above the diagonal
    for r, c, _ in chunks:
        assert 8 * c <= r


def test_bench_record_size_matches_the_header(layout):
    (*_, total), _ = layout
    import bench
    assert bench.REC_BYTES == total, "bench.py's record size differs from the layout header's REC_BYTES"
