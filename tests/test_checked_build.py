"""The range-checked build (-DATTN_CHECK): the same kernels with every copy
they issue checked against the tensor it reads (a failed check latches
ATTN_ERR_CHECK and the copy is skipped).  tests/checked_cases.py runs parity
cases of every kernel family against it in a process of its own; all must
match the oracle with no check failing.  The normal build compiles the
checks away (its register and spill counts are unchanged)."""
import os
import subprocess
import sys

import pytest

from causal_head_self_gb300 import build as _build

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_parity_cases_pass_every_range_check():
    _build.build(check=True)
    env = dict(os.environ, CHS_ATTN_CHECK="1")
    r = subprocess.run([sys.executable, os.path.join(HERE, "checked_cases.py")], env=env,
                       capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "backward_cases ok" in r.stdout
