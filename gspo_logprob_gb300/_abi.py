"""ctypes view of the C ABI declared in include/grpo_head.h.

Loads ``libgrpohead.so`` (built in-tree next to this file) and declares the
argument and return types of every entry point.  There is no fallback: if the
library is missing the import of the ops fails loudly.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_double, c_float, c_int32, c_int64, c_size_t, c_uint64, c_void_p

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libgrpohead.so")

# host status
GH_OK, GH_ERR_INVALID_ARG, GH_ERR_UNSUPPORTED, GH_ERR_WORKSPACE, GH_ERR_CUDA = range(5)
# device status bits
GH_DEV_TARGET_OOR, GH_DEV_NONFINITE, GH_DEV_TIMEOUT, GH_DEV_NO_ACTIVE, GH_DEV_BAD_SEQ = 1, 2, 4, 8, 16
DEV_BIT_NAMES = {1: "TARGET_OOR", 2: "NONFINITE", 4: "TIMEOUT", 8: "NO_ACTIVE", 16: "BAD_SEQ"}
# dtypes / reductions
GH_BF16, GH_FP32 = 0, 1
GH_TOKEN_MEAN, GH_SEQ_MEAN, GH_FIXED = 0, 1, 2
REDUCTIONS = {"token_mean": GH_TOKEN_MEAN, "seq_mean": GH_SEQ_MEAN, "fixed": GH_FIXED}
RATIO_LEVELS = {"token": 0, "sequence": 1}
NUM_KERNEL_KINDS = 18
NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024  # GH_NOALLOC_SCRATCH_BYTES


class GhHead(ctypes.Structure):
    _fields_ = [("N", c_int64), ("D", c_int64), ("V", c_int64), ("dtype", c_int32), ("row_tile", c_int32),
                ("H", c_void_p), ("W", c_void_p), ("targets", c_void_p), ("mask", c_void_p)]


class GhGrpo(ctypes.Structure):
    _fields_ = [("old_logp", c_void_p), ("ref_logp", c_void_p), ("adv", c_void_p), ("seq_id", c_void_p),
                ("num_seqs", c_int32), ("reduction", c_int32), ("eps_low", c_float), ("eps_high", c_float),
                ("beta", c_float), ("delta", c_float), ("norm", c_double), ("ratio_level", c_int32),
                ("reserved", c_int32), ("seq_policy", c_void_p), ("seq_kl", c_void_p), ("seq_count", c_void_p),
                ("num_clipped", c_void_p)]


# name -> (restype, argtypes)
SIGNATURES = {
    "grpo_head_forward_workspace_size": (c_size_t, [POINTER(GhHead)]),
    "grpo_head_backward_workspace_size": (c_size_t, [POINTER(GhHead)]),
    "grpo_head_backward_shard_workspace_size": (c_size_t, [POINTER(GhHead), c_int64]),
    "grpo_head_forward": (c_int32, [POINTER(GhHead), POINTER(GhGrpo), c_void_p, c_void_p, c_void_p, c_void_p,
                                    c_void_p, c_void_p, c_size_t, c_void_p]),
    "gspo_segment_workspace_size": (c_size_t, [c_int32]),
    "gspo_segment_loss": (c_int32, [c_int64, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int32, c_void_p,
                                    c_float, c_float, c_float, c_double, c_int32, c_void_p, c_void_p, c_void_p,
                                    c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "gspo_segment_partials": (c_int32, [c_int64, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int32,
                                        c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "gspo_segment_loss_from_partials": (c_int32, [c_int64, c_void_p, c_void_p, c_void_p, c_void_p, c_int32, c_int32,
                                                  c_void_p, c_void_p, c_void_p, c_float, c_float, c_float, c_double,
                                                  c_int32, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                                  c_void_p, c_void_p, c_size_t, c_void_p]),
    "grpo_head_backward": (c_int32, [POINTER(GhHead), c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int32,
                                     c_void_p, c_void_p, c_size_t, c_void_p]),
    "grpo_group_advantage": (c_int32, [c_void_p, c_int32, c_int32, c_float, c_void_p, c_void_p, c_void_p]),
    "grpo_head_forward_noalloc": (c_int32, [POINTER(GhHead), POINTER(GhGrpo), c_void_p, c_void_p, c_void_p,
                                            c_void_p, c_void_p, c_void_p]),
    "gh_vocab_shard_bounds": (c_int32, [c_int64, c_int32, c_int32, POINTER(c_int64), POINTER(c_int64)]),
    "gh_vocab_splits": (c_int64, [c_int64]),
    "grpo_head_logprob_shard": (c_int32, [POINTER(GhHead), c_int64, c_int64, c_void_p, c_void_p, c_void_p, c_void_p,
                                          c_void_p]),
    "grpo_logprob_merge": (c_int32, [c_int64, c_int64, c_int32, POINTER(c_int64), c_void_p, c_void_p, c_void_p,
                                     c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    "grpo_head_backward_shard": (c_int32, [POINTER(GhHead), c_int64, c_int64, c_void_p, c_void_p, c_void_p,
                                           c_void_p, c_void_p, c_int32, c_void_p, c_void_p, c_size_t, c_void_p]),
    "grpo_dh_merge": (c_int32, [c_int32, c_int64, c_int64, c_int32, c_void_p, c_void_p, c_void_p, c_void_p]),
    "grpo_loss_from_sequence_totals": (c_int32, [c_int32, c_void_p, c_void_p, c_void_p, c_int32, c_double, c_float,
                                                 c_void_p, c_void_p, c_void_p]),
    "gh_status_string": (c_char_p, [c_int32]),
    "gh_last_error": (c_char_p, []),
    "gh_abi_version": (c_int32, []),
    "gh_profile_enable": (None, [c_int32]),
    "gh_profile_reset": (None, []),
    "gh_profile_read": (c_int32, [c_int32, POINTER(c_int64), POINTER(c_double)]),
    "gh_launch_count": (c_int64, []),
    "gh_kernel_kind_name": (c_char_p, [c_int32]),
    "gh_timeout_probe": (c_int32, [c_void_p, c_uint64, c_void_p]),
}

_lib = None


def load(path: str = LIB_PATH):
    """Load the library once and declare its signatures; raise if it is absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"CUDA library not built: {path} is missing. Build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc with sm_103a).")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class GhError(RuntimeError):
    pass


def check(code: int, what: str) -> None:
    if code != GH_OK:
        lib = load()
        raise GhError(f"{what}: {lib.gh_status_string(code).decode()} ({lib.gh_last_error().decode()})")


def describe_status(word: int) -> str:
    names = [n for b, n in DEV_BIT_NAMES.items() if word & b]
    return "|".join(names) if names else "OK"
