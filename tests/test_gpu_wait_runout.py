"""Failure detection on the device: a bounded mbarrier wait that runs out.

Every mbarrier wait in the kernels gives up after a bounded number of cycles,
sets a bit in the device error word and lets the CTA finish, so that a stuck
pipeline reports an error instead of hanging the GPU.  This test exercises that
path safely: a test build of the library (-DDSR_TEST_WAIT_RUNOUT) shortens the
bound to ~1 ms and can stop the tensor-core decode kernel's producers from
issuing any copy, so the waits of the MMA and softmax warps run out while
nothing is in flight.  The call must return promptly with DS_DEVERR_WORKLIST
set, and the next normal call on the same device must match the oracle.  The
test build runs in a subprocess of its own (wait_runout_probe.py).
"""
import json
import os
import subprocess
import sys
import tempfile

import pytest

from ragged_blocked_kv_raggedbatch_gb300 import build as B

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_bounded_wait_runs_out_and_reports():
    out_dir = os.path.join(tempfile.gettempdir(), "ds_ragged_wait_runout_build")
    lib = B.build(out_dir=out_dir, extra_flags="-DDSR_TEST_WAIT_RUNOUT")
    r = subprocess.run([sys.executable, os.path.join(HERE, "wait_runout_probe.py"), lib],
                       capture_output=True, text=True, timeout=600)
    lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
    assert r.returncode == 0 and lines, r.stdout[-2000:] + r.stderr[-3000:]
    res = json.loads(lines[-1])
    assert res["ok"], res
    assert res["split_items"] > res["rows"]  # split rows: partials and the combine ran too
