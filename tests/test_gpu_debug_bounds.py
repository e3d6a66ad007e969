"""The bounds-checked build of the library, a stand-in for a memory checker (none can be run on
the GPU machines): small cases through every entry point must match the oracle with no access
outside the arrays of their calls, and a planted range shortfall must be reported (the check
skips the access and sets SV_ERR_BOUNDS; nothing traps). Runs in a child process, since a
process loads one build of the library."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_every_entry_point_stays_inside_its_arrays():
    import speculative_decoding_verification_rejection_gb300 as sv

    sv.build(debug=True)
    env = dict(os.environ, SPEC_VERIFY_DEBUG_BOUNDS="1")
    env.pop("SV_DEBUG_SHRINK", None)
    r = subprocess.run([sys.executable, os.path.join(HERE, "debug_bounds_check.py")], env=env,
                       capture_output=True, text=True, timeout=900)
    print(r.stdout[-3000:])
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-3000:]
    assert r.stdout.strip().splitlines()[-1] == "OK"
