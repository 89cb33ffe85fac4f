"""The guarded build: libmla compiled with MLA_GUARD checks every plain global load and store of its
kernels against the extent of the buffer it belongs to and records the first access that would
leave it (status word 0x3000 | site; the access is skipped).  It serves as an out-of-bounds
checker where no external memory checker can run: small cases of every call run through the
guarded library (a child process loads it) must match the oracle with no check firing."""
import os
import subprocess
import sys

import pytest

from mla_attention_gb300 import build

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_guarded_build_runs_every_call_clean():
    path = build.build(guard=True)
    r = subprocess.run([sys.executable, os.path.join(HERE, "guarded_cases.py"), path], capture_output=True,
                       text=True, timeout=900, cwd=os.path.dirname(HERE))
    assert r.returncode == 0 and "guarded ok" in r.stdout, (r.stdout[-3000:] + r.stderr[-3000:])
