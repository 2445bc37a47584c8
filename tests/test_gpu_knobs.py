"""Every tile / raster / block-width tuning setting computes the same result:
each setting runs in a child process (the knobs are read once per process)
and is checked against the fp64 oracle, including multi-block backward
vocabularies that exercise every dH accumulation mode."""
import os
import subprocess
import sys

import pytest

from gpu_helpers import gpu_lib  # noqa: F401

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))

SETTINGS = [
    {"GH_BWD_BLOCK_COLS": "512"},                                  # 6 blocks: dH store / add / add+cast
    {"GH_BWD_BLOCK_COLS": "512", "GH_FWD_PAIR": "0", "GH_DLOGITS_PAIR": "0", "GH_DH_PAIR": "0", "GH_DW_PAIR": "0"},
    {"GH_BWD_BLOCK_COLS": "1024", "GH_DH_MT": "2", "GH_DLOGITS_MT": "1", "GH_DW_MT": "1", "GH_DLOGITS_PAIR": "0",
     "GH_DH_PAIR": "0", "GH_DW_PAIR": "0"},
    {"GH_BWD_BLOCK_COLS": "768", "GH_DLOGITS_GROUP_M": "1", "GH_DH_GROUP_M": "3", "GH_DW_GROUP_M": "64"},
    {"GH_BWD_BLOCK_COLS": "768", "GH_DLOGITS_GROUP_M": "1", "GH_DH_GROUP_M": "3", "GH_DW_GROUP_M": "64",
     "GH_DLOGITS_PAIR": "0", "GH_DH_PAIR": "0", "GH_DW_PAIR": "0"},
    {"GH_BWD_BLOCK_COLS": "1280", "GH_DH_MT": "2", "GH_DH_CG": "2", "GH_DW_CG": "2", "GH_DLOGITS_CG": "2",
     "GH_DLOGITS_PAIR": "0", "GH_DH_PAIR": "0", "GH_DW_PAIR": "0"},
    {"GH_FWD_PAIR": "1", "GH_DLOGITS_PAIR": "1", "GH_DH_PAIR": "1", "GH_DW_PAIR": "1", "GH_BWD_BLOCK_COLS": "1024"},
    {"GH_FWD_PAIR": "0", "GH_DLOGITS_PAIR": "0", "GH_DH_PAIR": "0", "GH_DW_PAIR": "0"},
    {"GH_FWD_PAIR": "0", "GH_DLOGITS_PAIR": "1", "GH_DH_PAIR": "0", "GH_DW_PAIR": "1", "GH_BWD_BLOCK_COLS": "768"},
]


@pytest.mark.parametrize("env", SETTINGS, ids=lambda e: ",".join(f"{k}={v}" for k, v in e.items()))
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_tuning_settings_match_oracle(gpu_lib, env, dtype):
    full = dict(os.environ)
    full.update(env)
    r = subprocess.run([sys.executable, os.path.join(HERE, "knob_child.py"), dtype], env=full, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("ok")
