"""The TF32 rounding of the tensor-core kernels' self-written operands
(tc_common.cuh, tf32_rna_bits: add half a TF32 unit in the last place to the
fp32 bit pattern, clear the low 13 bits) against an independent definition:
of the two TF32 values that bracket x, the nearer one, ties away from zero.
The header function is compiled for the host with nvcc and run on edge cases
and random finite patterns."""
import os
import shutil
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "causal_gqa_attention_attn_gb300", "csrc")

_PROG = r"""
#include <stdio.h>
#include <stdlib.h>
#include "tc_common.cuh"
int main(int argc, char** argv) {
  FILE* fi = fopen(argv[1], "rb");
  FILE* fo = fopen(argv[2], "wb");
  uint32_t u;
  while (fread(&u, 4, 1, fi) == 1) {
    const uint32_t r = gqa::tc::tf32_rna_bits(u);
    fwrite(&r, 4, 1, fo);
  }
  fclose(fi);
  fclose(fo);
  return 0;
}
"""


def _reference(u):
    """Nearest of the two bracketing TF32 values, ties away from zero."""
    u = u.astype(np.uint32)
    sign = u & np.uint32(0x80000000)
    mag = u & np.uint32(0x7FFFFFFF)
    lo = mag & np.uint32(0xFFFFE000)
    hi = lo + np.uint32(0x2000)
    v = mag.view(np.float32).astype(np.float64)
    vlo = lo.view(np.float32).astype(np.float64)
    # past the largest binade the upper neighbour is 2^128 (rounding there
    # overflows to infinity, whose pattern is hi)
    vhi = np.where(hi == np.uint32(0x7F800000), 2.0 ** 128,
                   hi.view(np.float32).astype(np.float64))
    pick_hi = (vhi - v) <= (v - vlo)                # ties go up in magnitude
    return np.where(pick_hi, hi, lo) | sign


def test_tf32_rounding_matches_nearest_ties_away(tmp_path):
    nvcc = shutil.which("nvcc") or ("/usr/local/cuda/bin/nvcc"
                                    if os.path.exists("/usr/local/cuda/bin/nvcc") else None)
    if nvcc is None:
        pytest.skip("nvcc not available")
    src = tmp_path / "tf32.cu"
    src.write_text(_PROG)
    exe = tmp_path / "tf32"
    subprocess.run([nvcc, "-O2", "-I", CSRC, "-o", str(exe), str(src)], check=True)
    rng = np.random.default_rng(5)
    edge = np.array([0x00000000, 0x80000000, 0x00000001, 0x00001000, 0x00001FFF, 0x00002000,
                     0x007FFFFF, 0x00800000, 0x3F800000, 0x3F800FFF, 0x3F801000, 0x3F801001,
                     0x3F802000, 0x3F803000, 0x3FFFF000, 0x3FFFEFFF, 0xBF801000, 0xBFFFF000,
                     0x7F7FEFFF, 0x7F7FF000, 0x7F7FFFFF, 0xFF7FFFFF], dtype=np.uint32)
    rand = rng.integers(0, 2**32, size=200_000, dtype=np.uint64).astype(np.uint32)
    rand = rand[(rand & 0x7F800000) != 0x7F800000]          # finite patterns only
    u = np.concatenate([edge, rand])
    fin, fout = tmp_path / "in.bin", tmp_path / "out.bin"
    u.tofile(fin)
    subprocess.run([str(exe), str(fin), str(fout)], check=True)
    got = np.fromfile(fout, dtype=np.uint32)
    ref = _reference(u)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(hex(u[i]), hex(got[i]), hex(ref[i])) for i in bad[:5]]
    # spot values: 1 + 2^-11 is a tie (rounds up), 1 + 2^-11 - ulp rounds down
    assert got[np.nonzero(u == 0x3F801000)[0][0]] == 0x3F802000
    assert got[np.nonzero(u == 0x3F800FFF)[0][0]] == 0x3F800000
