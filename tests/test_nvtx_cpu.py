"""Every C-ABI call opens one NVTX range named after itself and closes it on
return (no GPU needed).  A small NVTX injection library (tests/native) records
the ranges; a child process loads it through NVTX_INJECTION64_PATH and makes
the host-argument-error calls of test_abi, which return before launching
anything."""
import inspect
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "native", "nvtx_recorder.c")


@pytest.fixture(scope="module")
def recorder(tmp_path_factory):
    out = str(tmp_path_factory.mktemp("nvtx") / "libnvtx_recorder.so")
    inc = "/usr/local/cuda/include"
    r = subprocess.run(["gcc", "-O1", "-shared", "-fPIC", "-I", inc, "-o", out, SRC, "-ldl"], capture_output=True,
                       text=True)
    if r.returncode != 0:
        pytest.skip("cannot build the NVTX recorder: " + r.stderr[-300:])
    return out


def test_every_call_opens_and_closes_its_range(recorder, tmp_path):
    log = tmp_path / "nvtx.log"
    env = dict(os.environ, NVTX_INJECTION64_PATH=recorder, FS_NVTX_LOG=str(log))
    code = ("import tests.test_abi as t; t.test_host_argument_errors_return_without_launching()")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = log.read_text().splitlines()
    pushes = [x.split(" ", 1)[1] for x in lines if x.startswith("push ")]
    pops = sum(1 for x in lines if x == "pop")
    assert pushes and pops == len(pushes)
    # ranges are not nested: every push is followed by its pop
    assert all(a.startswith("push ") and b == "pop" for a, b in zip(lines[0::2], lines[1::2]))
    from tests import test_abi
    src = inspect.getsource(test_abi.test_host_argument_errors_return_without_launching)
    called = set(re.findall(r"L\.(fs_[a-z0-9_]+)\(", src))
    launching = {n for n in called if not n.endswith(("_workspace_size", "_words"))}
    assert len(launching) >= 10 and launching == set(pushes)
