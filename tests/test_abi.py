"""CPU checks of the C ABI: the library builds, loads and exports every entry
point declared in include/grpo_head.h; the ctypes struct layouts match the C
ones; host-only calls (names, versions, workspace sizes, argument
validation) behave as documented.  No kernel is launched here."""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "grpo_head.h")


@pytest.fixture(scope="module")
def lib():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available to build the library")
    from gspo_logprob_gb300 import build
    build()
    from gspo_logprob_gb300 import _abi
    return _abi.load()


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \*]*?\b([a-z_][a-z0-9_]*)\s*\(", src, flags=re.M)
    return sorted(set(n for n in names if n not in ("defined",)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert "grpo_head_forward" in names and "gspo_segment_loss" in names and "grpo_head_backward" in names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in the header but not exported"
    from gspo_logprob_gb300 import _abi
    assert set(names) == set(_abi.SIGNATURES), "ctypes signatures and header declarations differ"


def test_struct_layout_matches_c(lib, tmp_path):
    gcc = shutil.which("gcc") or shutil.which("cc")
    if gcc is None:
        pytest.skip("no C compiler")
    prog = tmp_path / "layout.c"
    prog.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "grpo_head.h"\n'
        "int main(void){printf(\"%zu %zu %zu %zu %zu %zu %zu %zu\\n\", sizeof(gh_head), offsetof(gh_head, H),"
        " offsetof(gh_head, mask), sizeof(gh_grpo), offsetof(gh_grpo, num_seqs), offsetof(gh_grpo, norm),"
        " offsetof(gh_grpo, ratio_level), offsetof(gh_grpo, seq_count));return 0;}\n")
    exe = tmp_path / "layout"
    subprocess.run([gcc, "-std=c99", "-I", os.path.join(ROOT, "include"), str(prog), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    from gspo_logprob_gb300._abi import GhGrpo, GhHead
    want = [ctypes.sizeof(GhHead), GhHead.H.offset, GhHead.mask.offset, ctypes.sizeof(GhGrpo),
            GhGrpo.num_seqs.offset, GhGrpo.norm.offset, GhGrpo.ratio_level.offset, GhGrpo.seq_count.offset]
    assert got == want


def test_host_only_calls(lib):
    assert lib.gh_abi_version() == 106
    assert lib.gh_status_string(0) == b"GH_OK"
    assert lib.gh_status_string(3) == b"GH_ERR_WORKSPACE"
    assert lib.gh_kernel_kind_name(0) == b"fwd_logits_lse_tc"
    assert lib.gh_kernel_kind_name(99) == b""


def _head(N=1000, D=256, V=5000, dtype=0, row_tile=0, aligned=True):
    from gspo_logprob_gb300._abi import GhHead
    base = 0x10000 if aligned else 0x10004
    return GhHead(N=N, D=D, V=V, dtype=dtype, row_tile=row_tile, H=base, W=base, targets=base, mask=base)


def test_workspace_sizes(lib):
    h = _head(N=1000, D=256, V=5000)
    # forward: two [splits, N] fp32 partial arrays + zy [N]; splits = ceil(5000/256) = 20;
    # then the GRPO loss's four per-sequence arrays for max(64, N/8) = 125 sequences
    # and 256 bytes of counters
    fw = lib.grpo_head_forward_workspace_size(ctypes.byref(h))
    al = lambda x: (x + 255) // 256 * 256
    assert fw == 2 * al(20 * 1000 * 4) + al(1000 * 4) + 4 * al(125 * 4) + 256
    # backward (bf16): one block of all 5120 padded columns, no dH accumulator;
    # all 1000 rows would take 10.24 MB against 3/4 of N*V*2 = 7.5 MB, so the rows
    # go in two chunks of 512 (whole 256-row tiles)
    bw = lib.grpo_head_backward_workspace_size(ctypes.byref(h))
    assert bw == al(512 * 5120 * 2) + 256          # + the tile counter of the fused dH/dW launch
    assert bw <= 0.75 * 1000 * 5000 * 2
    # a vocabulary of two 16384-column blocks adds the fp32 dH accumulator of a chunk
    h3 = _head(N=1000, D=256, V=20000)
    assert lib.grpo_head_backward_workspace_size(ctypes.byref(h3)) == al(512 * 16384 * 2) + al(512 * 256 * 4) + 256
    # a wide vocabulary keeps all rows in one chunk
    h6 = _head(N=8192, D=4096, V=151936)
    assert lib.grpo_head_backward_workspace_size(ctypes.byref(h6)) == \
        al(8192 * 16384 * 2) + al(8192 * 4096 * 4) + 256
    # fewer rows than one tile: a single chunk whatever the ratio
    h2 = _head(N=64, D=64, V=500)
    assert lib.grpo_head_backward_workspace_size(ctypes.byref(h2)) == al(64 * 512 * 2) + 256
    # fp32, N = D = 1024, V = 4096: 1024-column blocks, all rows (4 MB of the 6.3 MB
    # budget); the 64 output tiles of each GEMM would run two K slices in parallel,
    # but two [1024, 1024] fp32 partials do not fit what is left, so none is allocated
    h4 = _head(N=1024, D=1024, V=4096, dtype=1)
    assert lib.grpo_head_backward_workspace_size(ctypes.byref(h4)) == al(1024 * 1024 * 4) + 256
    # tiny fp32 problem (N=256, V=500): 64-row chunks keep the block at half of N*V*2
    h7 = _head(N=256, D=64, V=500, dtype=1)
    assert lib.grpo_head_backward_workspace_size(ctypes.byref(h7)) == al(64 * 512 * 4) + 256
    # a large fp32 problem needs no parallel slices
    h5 = _head(N=8192, D=4096, V=4096, dtype=1)
    assert lib.grpo_head_backward_workspace_size(ctypes.byref(h5)) == al(8192 * 1024 * 4) + 256
    # a vocabulary shard sizes its chunks by the whole vocabulary and needs no dH accumulator
    hs = _head(N=1000, D=256, V=2560)
    assert lib.grpo_head_backward_shard_workspace_size(ctypes.byref(hs), 5000) == al(512 * 2560 * 2) + 256
    assert lib.grpo_head_backward_shard_workspace_size(ctypes.byref(hs), 2000) == 0      # V_total < V
    # invalid problem -> 0
    assert lib.grpo_head_forward_workspace_size(ctypes.byref(_head(D=12))) == 0


@pytest.mark.parametrize("kw,msg", [
    (dict(D=12), b"D % 8"),
    (dict(row_tile=96), b"row_tile"),
    (dict(dtype=7), b"dtype"),
    (dict(V=0), b"V="),
    (dict(aligned=False), b"aligned"),
])
def test_argument_validation(lib, kw, msg):
    h = _head(**kw)
    st = lib.grpo_head_forward(ctypes.byref(h), None, 0x100, 0x100, None, None, 0x100, 0x100, 1 << 30, None)
    assert st == 1  # GH_ERR_INVALID_ARG
    assert msg in lib.gh_last_error()


def test_workspace_too_small_is_reported(lib):
    h = _head()
    st = lib.grpo_head_forward(ctypes.byref(h), None, 0x100, 0x100, None, None, 0x100, 0x100, 16, None)
    assert st == 3  # GH_ERR_WORKSPACE


def test_no_gpu_fails_loudly(lib):
    # with a valid problem but no sm_103 device the call must refuse, not fall back
    try:
        import torch
        if torch.cuda.is_available():
            pytest.skip("a GPU is present")
    except ImportError:
        pass
    h = _head()
    st = lib.grpo_head_forward(ctypes.byref(h), None, 0x100, 0x100, None, None, 0x100, 0x100, 1 << 30, None)
    assert st == 2  # GH_ERR_UNSUPPORTED
    assert b"sm_103" in lib.gh_last_error()


def test_gspo_and_advantage_validation(lib):
    st = lib.gspo_segment_loss(10, 0x100, 0x100, None, 0x100, 0x100, 0, 0x100, 0.2, 0.2, 0.0, 1.0, 0, 0x100, None,
                               0x100, None, None, 0x100, None, 0, None)
    assert st == 1 and b"num_segments" in lib.gh_last_error()
    st = lib.gspo_segment_loss(10, 0x100, 0x100, None, 0x100, 0x100, 4, 0x100, 0.2, 0.2, 0.0, 0.0, 0, 0x100, None,
                               0x100, None, None, 0x100, None, 0, None)
    assert st == 1 and b"divisor" in lib.gh_last_error()
    st = lib.gspo_segment_loss(10, 0x100, 0x100, None, 0x100, 0x100, 4, 0x100, 0.2, 0.2, 0.1, 1.0, 0, 0x100, None,
                               0x100, None, None, 0x100, None, 0, None)
    assert st == 1 and b"ref_logp" in lib.gh_last_error()
    # a workspace smaller than gspo_segment_workspace_size is refused
    need = lib.gspo_segment_workspace_size(4)
    assert need > 0 and lib.gspo_segment_workspace_size(0) == 0
    st = lib.gspo_segment_loss(10, 0x100, 0x100, None, 0x100, 0x100, 4, 0x100, 0.2, 0.2, 0.0, 1.0, 0, 0x100, None,
                               0x100, None, None, 0x100, 0x10000, need - 1, None)
    assert st == 3 and b"GSPO workspace" in lib.gh_last_error()
    st = lib.grpo_group_advantage(0x100, 10, 4, 1e-4, 0x100, 0x100, None)
    assert st == 1 and b"multiple" in lib.gh_last_error()


def test_binding_imports_without_gpu():
    import gspo_logprob_gb300 as g
    assert callable(g.grpo_head_forward) and callable(g.grpo_head_backward)


def test_vocab_shard_bounds(lib):
    import gspo_logprob_gb300 as g
    assert [lib.gh_vocab_splits(v) for v in (0, 1, 256, 257, 5000, 151936)] == [0, 1, 1, 2, 20, 594]
    assert g.vocab_shard_bounds(5000, 2) == [(0, 2560), (2560, 2440)]
    b = g.vocab_shard_bounds(151936, 4)   # 594 splits of 256 -> 149, 149, 148, 148
    assert b == [(0, 38144), (38144, 38144), (76288, 37888), (114176, 37760)]
    for V, P in ((5000, 5), (151936, 7), (1, 1), (1025, 2)):
        b = g.vocab_shard_bounds(V, P)
        assert b[0][0] == 0 and sum(x[1] for x in b) == V
        assert all(x[0] % 256 == 0 for x in b)
        assert all(b[i][0] + b[i][1] == b[i + 1][0] for i in range(P - 1))
    st, ln = ctypes.c_int64(), ctypes.c_int64()
    assert lib.gh_vocab_shard_bounds(5000, 20, 0, ctypes.byref(st), ctypes.byref(ln)) == 0
    assert lib.gh_vocab_shard_bounds(5000, 21, 0, ctypes.byref(st), ctypes.byref(ln)) == 1  # more shards than splits


def test_shard_argument_validation(lib):
    h = _head(N=100, D=64, V=3000)
    # vocab_start not on the 256-column split grid
    assert lib.grpo_head_logprob_shard(ctypes.byref(h), 384, 5000, 0x100, 0x100, 0x100, 0x100, None) == 1
    # a middle shard that is not whole splits
    assert lib.grpo_head_logprob_shard(ctypes.byref(h), 0, 5000, 0x100, 0x100, 0x100, 0x100, None) == 1
    assert b"whole" in lib.gh_last_error()
    starts = (ctypes.c_int64 * 3)(0, 3000, 5000)
    assert lib.grpo_logprob_merge(100, 5000, 2, starts, 0x100, 0x100, 0x100, 0x100, 0x100, 0x100, 0x100, 0x100,
                                  None) == 1


# workloads (N, D, V, dtype) whose workspaces must stay below the bf16 [N, V]
# logits they never form: the five configurations, in both dtypes where the
# path exists, and the packed-GSPO shapes
_MEMORY_CASES = [
    ("tiny fp32 GRPO", 256, 64, 500, 1),
    ("tiny GRPO in bf16", 256, 64, 500, 0),
    ("selective logp bf16", 4096, 256, 5000, 0),
    ("selective logp fp32", 4096, 256, 5000, 1),
    ("bf16 GRPO small", 1024, 1024, 4096, 0),
    ("fp32 GRPO small", 1024, 1024, 4096, 1),
    ("bf16 GSPO packed", 16384, 2048, 32000, 0),
    ("bf16 8B-vocab micro-batch", 8192, 4096, 151936, 0),
]


@pytest.mark.parametrize("name,N,D,V,dtype", _MEMORY_CASES)
def test_extra_memory_below_logits(lib, name, N, D, V, dtype):
    # peak extra device memory of a forward + backward is the larger of the two
    # workspaces (the library allocates nothing else): at most 3/4 of N*V*2
    # (the method's memory claim is that [N, V] is never materialised)
    h = _head(N=N, D=D, V=V, dtype=dtype)
    fw = lib.grpo_head_forward_workspace_size(ctypes.byref(h))
    bw = lib.grpo_head_backward_workspace_size(ctypes.byref(h))
    ratio = max(fw, bw) / (N * V * 2)
    print(f"{name}: forward {fw} B, backward {bw} B, {ratio:.3f} of N*V*2")
    assert ratio <= 0.75 + 256 / (N * V * 2) + 1e-9
