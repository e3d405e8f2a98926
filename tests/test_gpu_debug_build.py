"""GPU: the FPD_DEBUG build (libfpd_debug.so).  Every entry point waits for its own kernels and returns their CUDA
error or device-side check as its status, so a bad input is reported by the call that consumed it instead of by a
later fpd_device_status.  Runs in a child process: the library is chosen when the package is imported."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import os, sys
import numpy as np
import torch
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))
import __graft_entry__ as g
g.build_debug()
os.environ["FPD_LIBRARY"] = "debug"
import block_diffusion_speculative_non_gb300 as pkg
assert pkg.LIB_PATH.endswith("libfpd_debug.so"), pkg.LIB_PATH
g.smoke()   # the small path, call by call, each synchronised and checked
import synth
s = synth.TINY
w = synth.make_weights(s, 77)
dr = pkg.Drafter(s, w, 1, 8, 32, device="cuda")
ctx = torch.zeros(1, dtype=torch.int32, device="cuda")
bad = torch.tensor([s.vocab + 5], dtype=torch.int32, device="cuda")
try:
    dr.draft_block(1, 8, ctx, bad, s.vocab - 1)
except pkg.FpdError as e:
    assert e.status == 6 and "device check 1" in str(e), str(e)
    print("debug build: bad anchor reported by fpd_draft_block:", e)
else:
    raise AssertionError("the debug build did not report the bad anchor")
assert pkg.fpd_device_status() == 1   # the check word is left for fpd_device_status too
dr.close()
"""


def test_debug_build_reports_device_checks_per_call():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ)
    env.pop("FPD_LIBRARY", None)
    r = subprocess.run([sys.executable, "-c", f"ROOT = {ROOT!r}\n" + SCRIPT], env=env, capture_output=True, text=True,
                       timeout=900)
    print(r.stdout[-2000:])
    assert r.returncode == 0, r.stderr[-4000:]
