"""The C ABI from a plain C host (tests/capi_loop.c, built here with gcc against
include/specdec.h and the in-tree libspecdec.so): every call of a back-to-back loop
returns SPECDEC_OK with the expected outputs, and the host cost of one chain call --
argument checks, pointer classification and the two launches -- stays small."""
import json
import os
import shutil
import subprocess
from pathlib import Path

import pytest

pytestmark = pytest.mark.gpu
ROOT = Path(__file__).resolve().parents[1]


def _cuda_home():
    for c in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if c and Path(c, "include", "cuda_runtime.h").exists():
            return Path(c)
    pytest.skip("CUDA toolkit headers not found")


@pytest.fixture(scope="module")
def capi_loop(built_library, tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not found")
    cuda = _cuda_home()
    lib = Path(built_library)
    exe = tmp_path_factory.mktemp("capi") / "capi_loop"
    libdirs = [d for d in (cuda / "lib64", cuda / "lib", cuda / "targets" / "sbsa-linux" / "lib",
                           cuda / "targets" / "x86_64-linux" / "lib") if d.exists()]
    cmd = ["gcc", "-O2", "-std=c11", "-D_POSIX_C_SOURCE=199309L", str(ROOT / "tests" / "capi_loop.c"),
           f"-I{ROOT / 'include'}", f"-I{cuda / 'include'}", "-o", str(exe), f"-L{lib.parent}", "-lspecdec",
           f"-Wl,-rpath,{lib.parent}"]
    for d in libdirs:
        cmd += [f"-L{d}", f"-Wl,-rpath,{d}"]
    cmd += ["-lcudart"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return exe


@pytest.mark.parametrize("B,g,V,limit_us", [(1, 4, 1000, 25.0), (64, 4, 32000, 25.0)])
def test_c_host_loop(capi_loop, B, g, V, limit_us):
    r = subprocess.run([str(capi_loop), str(B), str(g), str(V), "2000"], capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    d = json.loads(r.stdout.strip().splitlines()[-1])
    assert d["ok"]
    path = os.environ.get("SPECDEC_PARITY_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"workload": f"C host loop B={B} g={g} V={V}", **d}) + "\n")
    assert d["issue_us"] < limit_us, d
