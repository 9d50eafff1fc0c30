"""Host-side logic of bench.py on CPU: the key of the committed ncu traffic."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

CODE = """// header comment
__global__ void k(float* x) {  // trailing comment
  /* block
     comment */
  x[0] = 1.f;

}
"""


def test_code_digest_ignores_comments_and_blank_lines():
    edited = CODE.replace("header comment", "a different header").replace("trailing comment", "") + "\n\n// more\n"
    assert bench.code_digest([CODE]) == bench.code_digest([edited])


def test_code_digest_sees_code_changes():
    assert bench.code_digest([CODE]) != bench.code_digest([CODE.replace("1.f", "2.f")])
    assert bench.code_digest([CODE, CODE]) != bench.code_digest([CODE])

