"""The C ABI from plain C: tests/c_abi/verify_from_c.c allocates its device buffers with
cudaMalloc, calls dspark_schedule_pack, dspark_verify_scatter (compact) and dspark_verify
(cap-accept) on the legacy default stream, and compares every output with the C oracle on the
same seeded inputs (bit for bit). No Python or PyTorch is between the caller and the library."""
import os
import subprocess

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_plain_c_caller_matches_the_oracle(tmp_path):
    from speculative_decoding_ragged_gb300 import build
    import oracle
    lib = build.build()
    olib = oracle.build()
    nvcc = build.nvcc()
    exe = str(tmp_path / "verify_from_c")
    pkg, odir = os.path.dirname(lib), os.path.dirname(olib)
    cmd = [nvcc, "-O2", "-I", os.path.join(ROOT, "include"),
           os.path.join(HERE, "c_abi", "verify_from_c.c"), "-o", exe,
           "-L", pkg, "-ldspark", "-L", odir, "-ldspark_oracle",
           "-Xlinker", f"-rpath={pkg}", "-Xlinker", f"-rpath={odir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, run.stdout + run.stderr
    assert run.stdout.strip().endswith("ok"), run.stdout
    # a case that exercises the path: windows beyond the anchor, drafts accepted
    fields = dict(kv.split("=") for kv in run.stdout.split()[:4])
    print(run.stdout.splitlines()[0])
    assert int(fields["M"]) > 12 and int(fields["K*"]) > 0 and int(fields["accepted"]) > 12
