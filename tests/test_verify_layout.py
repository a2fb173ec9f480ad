"""Host logic of the batched verify step: the tile geometry of its GEMM steps and the layout of the
repacked weight blocks, compiled from the library's own header (quantized_gemv_gb300/csrc/mk_verify.h)
as plain C++ and checked against the model shape:

* segment packing: R rows of a CTA in S segments of KS inputs fill the MMA's 128 rows (S R = 128),
  every segment is a whole number of 64-column boxes, N = 16 S B rows (high and low parts of up to 8
  tokens) within the instruction's limit of 256, and the B operand fits the 96 KB staging buffer;
* the rows the CTAs own cover each matrix exactly (q|k|v 4,096, o_proj 1,024, gate/up 6,144 on
  96 CTAs, down 1,024);
* the blocks of one layer (step after step, CTA after CTA) tile its bytes without gap or overlap,
  and hold every weight once as a 16-bit value;
* the LM head: every CTA's rows fit its 128-row chunks.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "quantized_gemv_gb300", "csrc")

SRC = r"""
#define __host__
#define __device__
#define __forceinline__ inline
#include "mk_verify.h"
#include <cstdio>
int main() {
  using namespace mk;
  for (int s = 0; s < VS_COUNT; ++s) {
    const VStepGeom g = v_step_geom(s);
    std::printf("geom %d %d %d %d %d %d %d %zu\n", s, g.R, g.S, g.KS, g.KB, g.N, v_cols(s), v_step_bytes(s));
    for (int c = 0; c < V_GRID; ++c) std::printf("block %d %d %zu %d\n", s, c, v_block_offset(s, c), v_nbox(s, c));
  }
  std::printf("layer %zu\n", v_layer_bytes());
  std::printf("head %d %zu\n", v_head_chunks(151936), v_head_cta_bytes(151936));
  std::printf("consts %d %d %d %d %zu %d\n", VK, VN, V_GRID, V_GU_CTAS, V_BOX, V_HEAD_CHUNK);
  return 0;
}
"""

ROWS = {0: 4096, 1: 1024, 2: 6144, 3: 1024}   # q|k|v, o_proj, gate+up, down
COLS = {0: 1024, 1: 2048, 2: 1024, 3: 3072}
V_XB = 3 * 256 * 128                            # the staging buffer (down_proj's B operand)


@pytest.fixture(scope="module")
def layout(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    d = tmp_path_factory.mktemp("verify_layout")
    src, exe = d / "layout.cpp", d / "layout"
    src.write_text(SRC)
    subprocess.run([cxx, "-std=c++17", "-I", CSRC, "-I", os.path.join(ROOT, "include"), "-o", str(exe), str(src)],
                   check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    res = {"geom": {}, "block": {}}
    for line in out:
        f = line.split()
        if not f:
            continue
        if f[0] == "geom":
            s, R, S, KS, KB, N, K, nbytes = map(int, f[1:])
            res["geom"][s] = dict(R=R, S=S, KS=KS, KB=KB, N=N, K=K, bytes=nbytes)
        elif f[0] == "block":
            s, c, off, nbox = map(int, f[1:])
            res["block"][(s, c)] = (off, nbox)
        elif f[0] == "layer":
            res["layer"] = int(f[1])
        elif f[0] == "head":
            res["head_chunks"], res["head_cta_bytes"] = int(f[1]), int(f[2])
        elif f[0] == "consts":
            res["VK"], res["VN"], res["grid"], res["gu_ctas"], res["box"], res["chunk"] = map(int, f[1:])
    return res


def test_segment_packing_fills_the_mma(layout):
    for s, g in layout["geom"].items():
        assert g["S"] * g["R"] == 128, s                      # every MMA row is a weight row
        assert g["KS"] * g["S"] == g["K"] == COLS[s], s       # the segments split K exactly
        assert g["KS"] % 64 == 0 and g["KB"] == g["KS"] // 64, s
        assert g["N"] == layout["VN"] * g["S"] <= 256 and g["N"] % 16 == 0, s
        assert g["KB"] * g["N"] * 128 <= V_XB, s             # the B operand fits the staging buffer
    assert layout["VN"] == 2 * layout["VK"]                   # high and low parts of up to VK tokens


def test_rows_cover_each_matrix(layout):
    for s, g in layout["geom"].items():
        ctas = layout["gu_ctas"] if s == 2 else layout["grid"]
        assert g["R"] * ctas == ROWS[s], s
        assert sum(1 for c in range(layout["grid"]) if layout["block"][(s, c)][1] > 0) == ctas, s


def test_blocks_tile_the_layer(layout):
    spans = []
    for (s, c), (off, nbox) in layout["block"].items():
        if nbox:
            spans.append((off, off + nbox * layout["box"]))
    spans.sort()
    pos = 0
    for a, b in spans:
        assert a == pos, (a, pos)     # no gap, no overlap
        pos = b
    assert pos == layout["layer"]
    assert layout["layer"] == 2 * sum(ROWS[s] * COLS[s] for s in ROWS)  # every weight once, 16 bits
    for s, g in layout["geom"].items():
        assert g["bytes"] == 2 * ROWS[s] * COLS[s], s


def test_lm_head_chunks_hold_every_cta_row(layout):
    vocab, grid, chunk = 151936, layout["grid"], layout["chunk"]
    most = max((vocab * (c + 1)) // grid - (vocab * c) // grid for c in range(grid))
    assert layout["head_chunks"] * chunk >= most
    assert layout["head_cta_bytes"] == layout["head_chunks"] * chunk * 1024 * 2
