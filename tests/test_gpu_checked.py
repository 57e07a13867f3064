"""The range-checked build (-DDSA_CHECKED).  Every kernel of that build checks
the indices and offsets of its shared-memory, TMEM and global accesses before
using them; a failed check sets DSA_STATUS_CHECK_FAILED and skips the access
(it never traps).  These tests build it and run the small parity suite against
it in a child process: every parity test must pass, and the suite's module
fixture requires a zero status word, so no check may fail."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.fixture(scope="module")
def checked_lib():
    from sparse_attention_gemm_gb300 import build

    return build.build(checked=True)


def _child(args, lib, timeout=1200):
    env = dict(os.environ, DSA_LIB_PATH=lib)
    return subprocess.run([sys.executable, *args], cwd=ROOT, env=env, capture_output=True, text=True,
                          timeout=timeout)


def test_checked_library_is_the_one_loaded(checked_lib):
    code = ("import torch; from sparse_attention_gemm_gb300 import ops; ops.lib(); "
            "print([l.split()[-1] for l in open('/proc/self/maps') if 'libdsa' in l][0])")
    r = _child(["-c", code], checked_lib, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert os.path.samefile(r.stdout.strip().splitlines()[-1], checked_lib)


def test_parity_suite_on_checked_build(checked_lib):
    r = _child(["-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", os.path.join(HERE, "test_gpu_parity.py")],
               checked_lib)
    assert r.returncode == 0, (r.stdout[-3000:], r.stderr[-2000:])
