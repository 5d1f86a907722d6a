"""The bounds-checked build (-DPPS_CHECKED) on the GPU: every evaluator and
search runs bit-exact against the oracle and no kernel check fires.  The
checked library is built here and loaded in a process of its own."""
import json
import os
import subprocess
import sys

import pytest

from conftest import ROOT

pytestmark = pytest.mark.gpu


def test_checked_build_runs_clean():
    from pipeline_schedule_simulation_gb300 import build_lib
    build_lib.build(checked=True)
    env = dict(os.environ, PPSCHED_CHECKED="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "checked_cases.py")], env=env, cwd=ROOT,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res["checked"] is True          # the checked library was the one loaded
    assert res["failure"] == 0, hex(res["failure"])
    assert res["cases"] >= 40
