"""The bounds-checked build (libmk_bounds.so, compiled with MK_BOUNDS): every
checked access of the kernel -- the producer's bulk-copy sources and ring
destinations, the consumers' ring-stage reads, and the global loads and
stores of the queries, K/V rows, split-KV partials, residual stream, h,
tagged words, logits and argmax slots -- is tested against its buffer before
it happens, and a violation would record MK_ERR_BOUNDS (with SM, pc and op)
in the error word and skip the access.  These tests run the small model
through it in a fresh process (the binding loads it when MK_LIB=bounds) and
require the oracle's results with no bounds error, over several step kinds:
one step per launch, several steps per launch, a paged cache, race stress
and the per-phase launches."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import sys
sys.path.insert(0, %(root)r)
from decode_megakernel_sm_gb300 import _lib as L
import synth
from tests.harness import Run
assert L.lib()._name.endswith("libmk_bounds.so"), L.lib()._name
cfg = synth.CONFIGS["tiny"]
r = Run(cfg, seed=3)
for _ in range(3):
    r.step()                       # one step per launch, parity + appended K/V rows
r.multi_step(3)                    # three greedy steps in one launch
for mode in ("stream", "graph", "pdl"):
    r.step(mode)                   # per-phase launches
r.close()
r = Run(synth.custom(prefill=(40, 40), steps=4), seed=5, paged=16, stress=(2000, 7, 1))
for _ in range(3):
    r.step()                       # paged cache under race stress
r.close()
print("bounds ok")
"""


def test_bounds_build_runs_the_small_model_clean():
    env = dict(os.environ, MK_LIB="bounds")
    out = subprocess.run([sys.executable, "-c", SCRIPT % {"root": ROOT}], env=env, cwd=ROOT,
                         capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stdout[-3000:] + out.stderr[-3000:]
    assert "bounds ok" in out.stdout
