"""The bounds-checked build, libtreeverify_checked.so: the same sources
compiled with TV_CHECKED, in which every index a kernel computes is checked
before the access it guards and a failed check is recorded in a device word
(no trap).  The whole GPU parity suite runs again against it, in a child
process with TV_CHECKED=1, where an autouse fixture (tests/conftest.py) reads
the record after every test and fails the test if any check failed; and the
mechanism itself is tested with tv_debug_check_selftest, whose stores all lie
inside its buffer whichever build runs it."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SELFTEST_UNIT = 9  # the library unit (tv_api.cu)


@pytest.fixture(scope="module")
def tv():
    import speculative_decoding_tree_tv_gb300 as m
    return m


def run_selftest(tv, n, logical_n):
    buf = torch.full((n,), -1, dtype=torch.int32, device="cuda:0")
    stream = torch.cuda.current_stream().cuda_stream
    assert tv.lib.tv_debug_check_selftest(buf.data_ptr(), n, logical_n, stream) == tv.TV_OK
    torch.cuda.synchronize()
    return buf.cpu()


def test_selftest_in_this_build(tv):
    assert tv.check_take() == 0
    got = run_selftest(tv, 300, 100)
    site = tv.check_take()
    if tv.CHECKED:
        # the guarded stores past the logical length were skipped and recorded
        assert torch.equal(got[:100], torch.arange(100, dtype=torch.int32))
        assert (got[100:] == -1).all()
        assert site >> 16 == SELFTEST_UNIT and (site & 0xffff) > 0
        assert tv.check_take() == 0  # the record was cleared
    else:
        assert tv.lib.tv_checked_build() == 0
        assert torch.equal(got, torch.arange(300, dtype=torch.int32))
        assert site == 0
    # inside the logical length nothing is recorded in either build
    assert torch.equal(run_selftest(tv, 64, 64), torch.arange(64, dtype=torch.int32))
    assert tv.check_take() == 0


@pytest.mark.skipif(os.environ.get("TV_CHECKED", "0") not in ("", "0"),
                    reason="already running under the checked build")
def test_parity_suite_under_the_checked_build():
    env = dict(os.environ, TV_CHECKED="1")
    # every GPU test, this file's selftest included (this test skips itself there)
    cmd = [sys.executable, "-m", "pytest", "tests", "-m", "gpu", "-x", "-q", "-p",
           "no:cacheprovider"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    tail = (r.stdout + r.stderr)[-4000:]
    print(tail)
    assert r.returncode == 0, tail
    # the child really loaded the checked build
    probe = subprocess.run(
        [sys.executable, "-c",
         "import speculative_decoding_tree_tv_gb300 as tv; "
         "print(tv.library_path(), tv.lib.tv_checked_build())"],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert probe.returncode == 0, probe.stderr
    path, flag = probe.stdout.split()
    assert path.endswith("libtreeverify_checked.so") and flag == "1"
