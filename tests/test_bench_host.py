"""bench.py's host logic that decides whether the committed ncu counters still describe the kernel."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402

SRC = '''// Kernel 2: the split partial.
__device__ float f(float x) {  // scaled
  /* a block
     comment */
  asm volatile("mov.u64 %0, %%globaltimer; // not a comment" : "=l"(t));
  return x * 2.f;
}
'''


def test_comments_and_blank_lines_do_not_count():
    edited = SRC.replace("// Kernel 2: the split partial.", "// Kernel 2: the per-split partial,\n// reworded.\n\n")
    edited = edited.replace("/* a block\n     comment */", "/* another */")
    assert bench._code_only(edited) == bench._code_only(SRC)


def test_code_and_string_literals_count():
    assert bench._code_only(SRC.replace("x * 2.f", "x * 3.f")) != bench._code_only(SRC)
    # inline PTX lives in string literals: a "//" inside one is code, not a comment
    assert "// not a comment" in bench._code_only(SRC)
    assert bench._code_only(SRC.replace("%%globaltimer;", "%%clock64;")) != bench._code_only(SRC)

