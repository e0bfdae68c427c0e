"""The debug build with device-side bounds checks (libmoelora_checked.so,
compiled with -DMOELORA_DEVICE_CHECKS): the kernels check every index they
take from the align's tables before the access it guards.  The same layer
calls -- decode, tiny, the dense MLP, CTA-pair tiles, the 3-kernel align path
and the dense linear with split shrink items, each on a 0xFF-filled
workspace -- run in two child processes, one per library.  No check may fail
(status OK; the out-of-range id case reads BAD_INDEX from the align's own
check) and the outputs of the two builds must be bit-identical."""
import os
import subprocess
import sys

import pytest
import torch

from lora_mixture_experts_gb300 import build

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CHILD = os.path.join(ROOT, "tests", "_checked_child.py")


def _run(lib, out):
    env = dict(os.environ, MOELORA_LIBRARY=lib)
    r = subprocess.run([sys.executable, CHILD, out], env=env, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    return torch.load(out)


def test_checked_build_flags_nothing_and_matches_release(tmp_path):
    release = _run(build.build(), str(tmp_path / "release.pt"))
    checked = _run(build.build(checked=True), str(tmp_path / "checked.pt"))
    assert checked["library"].endswith("libmoelora_checked.so")
    assert release["library"].endswith("libmoelora.so")
    names = [n for n in checked if n != "library"]
    assert sorted(names) == sorted(n for n in release if n != "library") and len(names) == 8
    for name in names:
        out_c, st_c = checked[name]
        out_r, st_r = release[name]
        want = -6 if name == "bad_id" else 0
        assert st_c == want and st_r == want, (name, st_c, st_r)
        assert torch.equal(out_c, out_r), name
