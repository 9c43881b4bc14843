"""The device codec's quotient method, checked exhaustively on the host.

The GPU kernels form each codec quotient (v / block scale, amax / 6) from an
approximate reciprocal and one fused multiply-add refinement instead of a
division. `native/codec_quotient_check.c` (plain C, compiled here with gcc,
no contraction of separate multiplies and adds) checks that this gives the
e2m1 / e4m3 code of the correctly rounded quotient for every scale code, every
bf16 value in the codec's range and every reciprocal within three ulps of the
exact one; the GPU sweeps in test_gpu_edge_scales.py then hold the kernels
themselves to the oracle on the same cases.
"""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def _run(tmp_path, *defines):
    exe = tmp_path / ("check" + "".join(defines))
    subprocess.run(["gcc", "-O2", "-ffp-contract=off", *[f"-D{d}" for d in defines], "-o", str(exe),
                    os.path.join(HERE, "native", "codec_quotient_check.c"), "-lm"], check=True)
    return subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_refined_quotient_gives_the_correctly_rounded_codes(tmp_path):
    out = _run(tmp_path)
    assert out.returncode == 0, out.stdout + out.stderr
    # 126 scales x 7 reciprocals x both signs of every bf16 up to 9 d; 7 x 32640 block maxima
    assert out.stdout.strip() == "e2m1 pairs 29595412 mismatches 0; e4m3 scales 228480 mismatches 0", out.stdout


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_check_rejects_the_unrefined_product(tmp_path):
    out = _run(tmp_path, "WITHOUT_REFINEMENT")
    assert out.returncode == 1 and "e2m1 mismatch" in out.stdout and "e4m3 mismatch" in out.stdout, out.stdout
