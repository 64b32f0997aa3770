"""The oracle's number conversions against formulations of their own over every
binary32 bit pattern (tests/host/conversions_brute.c, built here with gcc and
oracle/h3q_oracle.c): bf16 rounding and the E2M1 code of every non-NaN value,
and the E4M3 scale code of every 256th value s >= 0 and of every value within
256 ulps of one of its decision points; and the SiLU exponential exp_c within 2
ulp of binary64 exp for every binary32 z in [-104, 88.7].  `conversions_brute full`
checks E4M3 on every s >= 0 as well (minutes of CPU time: not part of this suite)."""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_conversions_every_binary32(tmp_path):
    exe = str(tmp_path / "conversions_brute")
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                    os.path.join(HERE, "host", "conversions_brute.c"),
                    os.path.join(ROOT, "oracle", "h3q_oracle.c"), "-o", exe, "-lm", "-pthread"], check=True)
    res = subprocess.run([exe], capture_output=True, text=True, timeout=900)
    assert res.returncode == 0, res.stdout + res.stderr
    assert "bf16 mismatches 0 e2m1 mismatches 0" in res.stdout
    assert "e4m3 (sampled and near every decision point) mismatches 0" in res.stdout
    assert "exp_c outside 2 ulp 0 " in res.stdout
