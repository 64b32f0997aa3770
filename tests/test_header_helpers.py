"""The inline size and offset helpers of include/h3q.h, compiled with gcc as a
C program and checked against the oracle's layout functions, and the Python
mirror of the row-tile offset used by the host-buffer pipeline."""
import os
import subprocess

import numpy as np
import pytest

import oracle
from nvfp4_activation_quantize_gb300.host import scale_offset_of_row_tile

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CASES = [(1, 64), (127, 64), (128, 128), (129, 256), (300, 7168), (65280, 7168), (65280, 18944),
         (300000, 7168)]

PROGRAM = r"""
#include <stdio.h>
#include <inttypes.h>
#include "h3q.h"
int main(void) {
    int64_t rows, cols, row0;
    while (scanf("%" SCNd64 " %" SCNd64 " %" SCNd64, &rows, &cols, &row0) == 3)
        printf("%" PRId64 " %" PRId64 " %" PRId64 " %" PRId64 "\n", h3q_padded_rows(rows),
               h3q_scale_bytes(rows, cols), h3q_code_bytes(rows, cols),
               h3q_scale_offset_of_row_tile(row0, cols));
    return 0;
}
"""


@pytest.fixture(scope="module")
def helper_bin(tmp_path_factory):
    d = tmp_path_factory.mktemp("hdr")
    src, exe = d / "h.c", d / "h"
    src.write_text(PROGRAM)
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe)], check=True)
    return str(exe)


def test_header_helpers_match_the_oracle_layout(helper_bin):
    lines, want = [], []
    for rows, cols in CASES:
        for row0 in sorted({0, 128, (rows - 1) // 128 * 128}):
            lines.append(f"{rows} {cols} {row0}")
            # the first scale of row row0 sits at the start of its row tile's atoms
            want.append((oracle.padded_rows(rows), oracle.padded_rows(rows) * cols // 16,
                         rows * cols // 2, oracle.scale_offset(row0, 0, cols)))
    out = subprocess.run([helper_bin], input="\n".join(lines) + "\n", capture_output=True,
                         text=True, check=True).stdout.split("\n")
    got = [tuple(int(v) for v in line.split()) for line in out if line]
    assert got == want


@pytest.mark.parametrize("rows,cols", [(300, 1024), (1000, 2048), (65280, 7168)])
def test_row_tiles_are_contiguous_ranges(rows, cols):
    """Every scale of rows [r0, r0 + 128k) lies in [tile offset of r0, tile offset of
    r0 + 128k): the property that lets a chunk's scales be copied as one range."""
    pad = oracle.padded_rows(rows)
    for r0, r1 in ((0, 128), (128, min(pad, 384)), (pad - 128, pad)):
        offs = oracle.scale_offsets(np.arange(r0, r1), cols)
        lo, hi = scale_offset_of_row_tile(r0, cols), scale_offset_of_row_tile(r1, cols)
        assert offs.min() == lo and offs.max() == hi - 1
        assert np.unique(offs).size == hi - lo


WORKSPACE_PROGRAM = r"""
#include <stdio.h>
#include <inttypes.h>
#include "h3q.h"
int main(void) {
    int64_t chunk, cols, rows, frames;
    while (scanf("%" SCNd64 " %" SCNd64 " %" SCNd64 " %" SCNd64, &chunk, &cols, &rows, &frames) == 4)
        printf("%" PRId64 "\n", h3q_host_workspace_bytes(chunk, cols, rows, (int)frames));
    return 0;
}
"""


def test_host_workspace_bytes_header_and_python_agree(tmp_path):
    from nvfp4_activation_quantize_gb300 import host_workspace_bytes

    src, exe = tmp_path / "w.c", tmp_path / "w"
    src.write_text(WORKSPACE_PROGRAM)
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe)], check=True)
    cases = [(128, 64, 1, 1), (8192, 7168, 65280, 1), (8192, 7168, 65280, 0), (256, 1088, 1000, 1),
             (384, 18944, 5, 0)]
    out = subprocess.run([str(exe)], input="".join(f"{c} {k} {r} {f}\n" for c, k, r, f in cases),
                         capture_output=True, text=True, check=True).stdout.split()
    assert [int(v) for v in out] == [host_workspace_bytes(c, k, r, bool(f)) for c, k, r, f in cases]
    # three slots of x, codes and scales (each rounded up to 256 bytes), then the frames
    assert host_workspace_bytes(8192, 7168, 65280, True) == 3 * (8192 * 7168 * (2 + 0.5 + 1 / 16)) + 65280 * 4
