"""The single-CTA conv kernel on the shapes the CTA-pair (tcgen05 cta_group::2)
kernel takes by default: the conv tests again with VAE_CONV_CTA_PAIR=0, in a
child process because the library reads the switch once per process."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_single_cta_conv_matches_oracle():
    env = dict(os.environ, VAE_CONV_CTA_PAIR="0")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_gpu_conv.py"), "-k", "not full_size"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
