"""Host-compiled checks of the kernels' own arithmetic helpers (no GPU)."""
import os
import subprocess

from allreduce_residual_rmsnorm_gb300 import build as BUILD

HERE = os.path.dirname(os.path.abspath(__file__))


def test_double_float_sum_of_squares_is_correctly_rounded(tmp_path):
    exe = tmp_path / "df_check"
    subprocess.check_call([BUILD.nvcc(), "-O2", "-std=c++17", "-I", BUILD.INCLUDE, "-I", BUILD.CSRC,
                           os.path.join(HERE, "host_df_check.cu"), "-o", str(exe)])
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
