"""Programmatic dependent launch (VAE_PDL=1, opt-in): every kernel waits for
its predecessor grid before touching global memory, so results must not change.
The decoder, attention and conv parity tests run again in a child process with
the switch on (the library reads it once per process)."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_parity_with_programmatic_dependent_launch():
    env = dict(os.environ, VAE_PDL="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_gpu_decoder.py"),
                        os.path.join(ROOT, "tests", "test_gpu_attention.py"),
                        "-k", "tiny or banded_decode_is or graph or mid_attention or peaked"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
