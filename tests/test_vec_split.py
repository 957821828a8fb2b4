"""The head/body/tail splitter behind the 16-byte vector loads of targets and LSE,
pinned to the worked example in the TransformerEngine pull request (#995)."""
import json
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "linear_cross_entropy_tcgen05_gb300", "csrc")

HARNESS = r"""
#include <stdio.h>
#include <stdlib.h>
#include "vec_split.h"
int main(int argc, char** argv) {
  long long start = atoll(argv[1]), len = atoll(argv[2]);
  int eb = atoi(argv[3]);
  flce_vec_split s = flce_split_for_vectors(start, len, eb);
  printf("%lld %lld %lld\n", (long long)s.head, (long long)s.body, (long long)s.tail);
  return 0;
}
"""


@pytest.fixture(scope="module")
def splitter(tmp_path_factory):
    cc = shutil.which("gcc") or shutil.which("cc")
    if not cc:
        pytest.skip("no C compiler")
    d = tmp_path_factory.mktemp("split")
    src = d / "h.c"
    src.write_text(HARNESS)
    exe = d / "h"
    subprocess.run([cc, "-O1", "-I", CSRC, str(src), "-o", str(exe)], check=True)

    def run(start, length, eb):
        out = subprocess.run([str(exe), str(start), str(length), str(eb)], capture_output=True, text=True,
                             check=True).stdout.split()
        return tuple(int(v) for v in out)

    return run


def test_transformer_engine_worked_example(splitter):
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "te_aligned_split.json")))
    n = g["row_length"]
    for r in g["rows"]:
        assert splitter(r["row"] * n, n, g["elem_bytes"]) == (r["head"], r["body"], r["tail"])


@pytest.mark.parametrize("eb", [1, 2, 4, 8])
def test_split_covers_the_run_with_aligned_vectors(splitter, eb):
    per = 16 // eb
    for start in range(0, 3 * per):
        for length in (0, 1, per - 1, per, per + 1, 5 * per + 3):
            h, b, t = splitter(start, length, eb)
            assert h + b + t == length and min(h, b, t) >= 0
            assert b % per == 0
            if b:
                assert (start + h) % per == 0
            assert h < per and t < per or b == 0
