"""The other draft launch paths (chosen once per process by environment
variables): the two-pass tensor-core kernel, one launch per pass, the
CUDA-core path, the 128-row fused tile at small batches too, and each stage
ring of the fused tile at every batch, each against the fp64 oracle in a child
process."""
import os
import subprocess
import sys

import pytest

from gpu_common import require_gpu

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import synth
from oracle.draft import draft as oracle_draft
from parity import compare_draft, gpu_np, np_inputs, rtol_for
from gpu_common import check_no_error, gpu_draft
for B, G, V, r, H in [(130, 5, 8200, 128, 16), (5, 4, 4104, 64, 24), (1, 3, 8200, 256, 16),
                     (600, 3, 4104, 256, 8)]:
    wl = synth.Workload("paths", B, G, V, H, r, "bf16", "mixed", synth.SCHED_GREEDY, "tiny", seed=11)
    inp = synth.make_inputs(wl, "cuda", with_target=False)
    out, ws = gpu_draft(inp)
    compare_draft(gpu_np(out), oracle_draft(**np_inputs(inp)), rtol_for("bf16"))
    check_no_error(ws)
print("ok")
"""


@pytest.mark.parametrize("env", [{"DSPARK_DRAFT_LAUNCH": "two_pass"}, {"DSPARK_DRAFT_LAUNCH": "per_pass"},
                                 {"DSPARK_DRAFT_PATH": "cuda_core"}, {"DSPARK_DRAFT_FORM": "wide"},
                                 {"DSPARK_FUSED_RING": "w2"}, {"DSPARK_FUSED_RING": "u"}])
def test_draft_launch_paths(env):
    require_gpu()
    code = CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"))
    res = subprocess.run([sys.executable, "-c", code], env={**os.environ, **env}, cwd=ROOT, capture_output=True,
                         text=True, timeout=600)
    assert res.returncode == 0 and res.stdout.strip().endswith("ok"), res.stdout[-2000:] + res.stderr[-4000:]
