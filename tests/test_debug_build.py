"""The bounds-checked debug build (libbi_debug.so, BI_LIBRARY=debug) on the GPU:
a failed check is recorded in the device status word and its access skipped
(no trap, no fault), and on valid inputs every kernel gives the same bits as
the release build with no check failing. compute-sanitizer is closed on the
GPUs this library is tested on; these checks stand in for its bounds checking."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


def run(code_or_script, debug, *args):
    env = dict(os.environ)
    env.pop("BI_LIBRARY", None)
    if debug:
        env["BI_LIBRARY"] = "debug"
    cmd = [sys.executable, os.path.join(HERE, code_or_script)] if code_or_script.endswith(".py") else \
        [sys.executable, "-c", code_or_script]
    r = subprocess.run(cmd + list(args), capture_output=True, text=True, env=env, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


PROBE = """
import json, sys
sys.path.insert(0, %r)
import invariant_deterministic_bi_gb300 as bi
bi.load()
out = {"debug": bi.debug_build()}
bi.check_bounds(5, 10)
out["inside"] = bi.status_string(bi.device_status())
bi.check_bounds(12, 10)
out["outside"] = bi.status_string(bi.device_status())
out["line"] = bi.last_bounds_line()
out["after"] = bi.status_string(bi.device_status())
print(json.dumps(out))
""" % os.path.dirname(HERE)


def test_failed_check_is_recorded_and_skipped():
    from invariant_deterministic_bi_gb300 import _build
    _build.build(debug=True)
    d = run(PROBE, debug=True)
    assert d["debug"] is True
    assert d["inside"] == "BI_OK"
    assert d["outside"] == "BI_ERR_BOUNDS" and d["line"] > 0
    assert d["after"] == "BI_OK"                      # reading the status cleared it
    r = run(PROBE, debug=False)                       # the release build compiles the check away
    assert r["debug"] is False and r["outside"] == "BI_OK"


def test_debug_and_release_builds_give_the_same_bits():
    from invariant_deterministic_bi_gb300 import _build
    _build.build(debug=True)
    rel = run("_debug_ops.py", debug=False)
    dbg = run("_debug_ops.py", debug=True)
    assert rel.pop("debug_build") is False and dbg.pop("debug_build") is True
    assert dbg["status"] == "BI_OK", "a bounds check failed on valid inputs"
    assert dbg == rel
