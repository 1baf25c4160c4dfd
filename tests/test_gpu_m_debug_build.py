"""The bounds-checked debug build (-DMOE_DEBUG: indices read from the schedule
arrays and the GEMMs' scale-atom addresses are checked before use, a failed
check recorded as MOE_ERR_BOUNDS).  With compute-sanitizer closed on this
pool, this build is the memory check of the indexing-heavy kernels: on every
reduced workload -- BF16 and MXFP8, forward and backward, the dispatch ring
and NVFP4 -- no check fires, and every output is bitwise the release build's."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def _run(env_lib):
    env = dict(os.environ)
    env.pop("MOE_GB300_LIB", None)
    if env_lib:
        env["MOE_GB300_LIB"] = env_lib
    r = subprocess.run([sys.executable, os.path.join(HERE, "debug_build_workloads.py")], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_debug_build_fires_no_check_and_changes_no_bit():
    from mixture_experts_layer_device_gb300 import build
    dbg = build.build(debug=True)
    rel = _run(None)
    deb = _run(dbg)
    assert deb["lib"] == dbg and rel["lib"] != dbg
    for name, res in rel.items():
        if name == "lib":
            continue
        for key, val in res.items():
            if key.endswith("_status"):
                assert val == 0 and deb[name][key] == 0, (name, key, deb[name][key])
            else:
                assert deb[name][key] == val, (name, key)
