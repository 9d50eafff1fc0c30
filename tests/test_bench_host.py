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



def _bench_reference(rank, world):
    import subprocess

    env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
               MASTER_ADDR="127.0.0.1", MASTER_PORT="29555")
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                           "--warmup", "3"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)


def test_reference_arm_prints_on_rank_0_only():
    """Under a two-rank launch the oracle arm runs on rank 0 alone, which
    prints one JSON line; rank 1 exits 0 without output."""
    import json

    r1 = _bench_reference(1, 2)
    assert r1.returncode == 0 and r1.stdout.strip() == ""
    r0 = _bench_reference(0, 2)
    assert r0.returncode == 0, r0.stderr
    lines = [ln for ln in r0.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
