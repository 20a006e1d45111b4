"""Concurrent first calls of the GEMM C ABI from several host threads (each on its own
stream), in a fresh process so that the library's per-device set-up is reached by all of
them at once; every output checked bit for bit against the oracle (tests/threads_child.py)."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_concurrent_first_calls_from_host_threads():
    r = subprocess.run([sys.executable, os.path.join(HERE, "threads_child.py")], capture_output=True,
                       text=True, timeout=900, cwd=os.path.dirname(HERE))
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-4000:]
    assert r.stdout.strip().startswith("ok")
