"""Host check of the tensor-core sweeps' persistent schedules, dense and under the causal and band pair
masks (torchpairwise guide, Score Expressions): tests/host/sched_check.cu includes the schedule header the
kernels use, runs every CTA's tile cursor over 7200 shapes, masks and band widths, and checks that every
tile holding a kept pair is visited once, every row block gets a tile, the partial slots are distinct and
each merge reads exactly the CTAs that met its row block; and the same for the upper triangle of tiles
that the X = Y log-sum-exp forward sweeps. CPU only: nvcc compiles it as host code."""
import os
import subprocess

from lazy_score_matrix_gb300 import build

HERE = os.path.dirname(os.path.abspath(__file__))


def test_schedules_visit_every_kept_tile_once(tmp_path):
    exe = str(tmp_path / "sched_check")
    src = os.path.join(HERE, "host", "sched_check.cu")
    subprocess.run([build.nvcc(), "-std=c++17", "-O2", *build.ARCH, "-o", exe, src], check=True,
                   capture_output=True, text=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "7200 schedules, " in r.stdout and " triangles, 0 failures" in r.stdout
