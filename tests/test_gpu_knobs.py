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
    {"GH_BWD_FUSED": "0", "GH_BWD_BLOCK_COLS": "512"},            # dH and dW as two pair launches per block
    {"GH_FWD_DYNAMIC": "1", "GH_BWD_BLOCK_COLS": "768"},           # forward tiles on demand
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


def _child(env, dtype="bf16"):
    full = dict(os.environ)
    full.update(env)
    r = subprocess.run([sys.executable, os.path.join(HERE, "knob_child.py"), dtype], env=full, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    words = r.stdout.split()
    return dict(x.split("=", 1) for x in words if "=" in x)


def test_backward_bits_do_not_depend_on_kernel_variant(gpu_lib):
    # a tile is always one chain of MMAs over K in the same order, whichever
    # kernel computes it: the fused dH/dW launch with dynamically handed-out
    # tiles, two pair launches, or the single-CTA kernels give the same bits
    # for the same vocabulary block width
    base = _child({"GH_BWD_BLOCK_COLS": "512"})
    unfused = _child({"GH_BWD_BLOCK_COLS": "512", "GH_BWD_FUSED": "0"})
    single = _child({"GH_BWD_BLOCK_COLS": "512", "GH_DLOGITS_PAIR": "0", "GH_DH_PAIR": "0", "GH_DW_PAIR": "0"})
    assert base == unfused == single, (base, unfused, single)
    # dW does not depend on the block width either (each element's K runs over the tokens)
    wide = _child({"GH_BWD_BLOCK_COLS": "1024"})
    assert wide["dW"] == base["dW"]


def test_forward_bits_do_not_depend_on_raster(gpu_lib):
    # the forward's raster group only changes which tiles run together; every
    # tile's partial and the fixed-order merge are the same
    base = _child({})
    for g in ("1", "3", "0"):
        other = _child({"GH_FWD_GROUP_M": g})
        assert (other["lse"], other["logp"]) == (base["lse"], base["logp"]), g


def test_forward_bits_do_not_depend_on_epilogue_groups(gpu_lib):
    # one or two groups of epilogue warps in the forward's CTA-pair kernel only
    # change how many tiles' epilogues run at once; every row's arithmetic is
    # the same (D = 192 here, so the default is two groups)
    base = _child({})
    for g in ("1", "2"):
        other = _child({"GH_FWD_EPI_GROUPS": g})
        assert (other["lse"], other["logp"]) == (base["lse"], base["logp"]), g


def test_forward_bits_do_not_depend_on_tile_hand_out(gpu_lib):
    # tiles taken on demand from a counter (the default for long K) or dealt
    # round-robin (the default here, D = 192): each tile is the same MMA chain
    # and epilogue, whichever pair computes it
    base = _child({"GH_FWD_DYNAMIC": "0"})
    for env in ({"GH_FWD_DYNAMIC": "1"}, {"GH_FWD_DYNAMIC": "1", "GH_FWD_GROUP_M": "3"}):
        other = _child(env)
        assert (other["lse"], other["logp"]) == (base["lse"], base["logp"]), env
