"""The bounds-checked build (-DNVFP4_CHECKED): on cases that reach every
instrumented kernel it records no failed check and gives the normal build's
outputs bit for bit; its check mechanism records an index outside its range
(a self-test that accesses nothing)."""
import json
import os
import subprocess
import sys

import pytest

import nvfp4_block_scale_gb300 as nv
from nvfp4_block_scale_gb300.build import build

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def run(which: str) -> dict:
    r = subprocess.run([sys.executable, os.path.join(HERE, "checked_cases.py"), which], capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_checked_build_matches_and_records_nothing():
    build()
    nv.checked_library_path(build=True)
    normal, checked = run("normal"), run("checked")
    assert normal["checked_build"] == 0 and checked["checked_build"] == 1
    assert checked["digests"] == normal["digests"]
    for k in ("start", "single", "deferred", "grouped", "selftest_inside"):
        assert checked["sites"][k] == 0, (k, hex(checked["sites"][k]))
    assert checked["sites"]["selftest_outside"] == 0x0001
    assert all(v == 0 for v in normal["sites"].values())  # the normal build records nothing
