"""Thin torch-facing binding of the C ABI (argument marshalling only).

Every function takes CUDA tensors, allocates its outputs and scratch space
with torch (device memory is the only thing torch provides here), and calls
the library entry point of the same name on the current CUDA stream.  All
arithmetic runs in the library's kernels; there is no CPU or framework
fallback.

Device-side status: each call returns (or fills) an int32 status tensor; use
``raise_on_status`` to read it (a host synchronisation) and raise on errors.
"""
from __future__ import annotations

import ctypes
import functools
from typing import Optional

import torch

from . import _abi
from ._abi import GhGrpo, GhHead

_BF16 = torch.bfloat16
_F32 = torch.float32


def _lib():
    return _abi.load()


_NVTX_OK = [None]  # None: not tried yet


def _nvtx_usable() -> bool:
    if _NVTX_OK[0] is None:
        try:
            torch.cuda.nvtx.range_push("gh.probe")
            torch.cuda.nvtx.range_pop()
            _NVTX_OK[0] = torch.cuda.is_available()
        except Exception:  # a torch build without NVTX: no ranges
            _NVTX_OK[0] = False
    return _NVTX_OK[0]


def _nvtx(fn):
    """Bracket a binding entry point with an NVTX range of its name, so a
    profiler timeline groups each call's kernels (no cost without a profiler)."""
    name = "gh." + fn.__name__

    @functools.wraps(fn)
    def wrapped(*args, **kwargs):
        if not _nvtx_usable():
            return fn(*args, **kwargs)
        torch.cuda.nvtx.range_push(name)
        try:
            return fn(*args, **kwargs)
        finally:
            torch.cuda.nvtx.range_pop()
    return wrapped


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(dev: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _need(t: torch.Tensor, name: str, dtype=None, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t


class _Workspace:
    """Grow-only scratch buffer per device, reused by consecutive calls.

    Calls whose GPU work overlaps on different streams must not share it (pass
    ``workspace=``).  Used from several streams one after the other, the buffer
    is marked as in use on each of them (``record_stream``), so that when it is
    replaced by a larger one torch's caching allocator does not hand its memory
    to other work before the kernels queued on those streams have finished."""

    def __init__(self):
        self._buf = {}

    def get(self, dev: torch.device, nbytes: int) -> torch.Tensor:
        key = (dev.type, dev.index)
        cur = torch.cuda.current_stream(dev)
        entry = self._buf.get(key)
        if entry is None or entry[0].numel() < nbytes:
            b = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
            entry = (b, {cur.cuda_stream})
            self._buf[key] = entry
        b, seen = entry
        if cur.cuda_stream not in seen:
            b.record_stream(cur)
            seen.add(cur.cuda_stream)
        return b

    def clear(self):
        self._buf.clear()


WORKSPACE = _Workspace()

_MAX_SEGMENTS = 16384
_SEAM_WS = {}


def _seam_workspace(dev: torch.device) -> torch.Tensor:
    """Scratch of the GSPO seam calls: one buffer per device, sized for the
    most segments a call takes, allocated once (its address never changes, so
    CUDA-graph captures of these calls stay valid).  Calls that overlap on
    different streams must pass their own ``workspace=``."""
    key = (dev.type, dev.index)
    b = _SEAM_WS.get(key)
    if b is None:
        b = torch.empty(int(_lib().gspo_segment_workspace_size(_MAX_SEGMENTS)), dtype=torch.uint8, device=dev)
        _SEAM_WS[key] = b
    return b


def _seam_ws(dev, num_segments: int, workspace: Optional[torch.Tensor]):
    nbytes = int(_lib().gspo_segment_workspace_size(int(num_segments)))
    ws = _caller_workspace(workspace, nbytes) if workspace is not None else _seam_workspace(dev)
    return ws, nbytes


def _caller_workspace(ws: torch.Tensor, nbytes: int) -> torch.Tensor:
    if not ws.is_cuda or not ws.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    if ws.numel() * ws.element_size() < nbytes:
        raise ValueError(f"workspace holds {ws.numel() * ws.element_size()} bytes; the call needs {nbytes}")
    return ws


def make_head(H: torch.Tensor, W: torch.Tensor, targets: torch.Tensor, mask: torch.Tensor,
              row_tile: int = 0) -> GhHead:
    _need(H, "H")
    _need(W, "W", dtype=H.dtype)
    if H.dtype not in (_BF16, _F32):
        raise TypeError("H/W must be bfloat16 or float32")
    if H.dim() != 2 or W.dim() != 2 or H.shape[1] != W.shape[1]:
        raise ValueError("H must be [N, D] and W [V, D]")
    N, D = H.shape
    V = W.shape[0]
    _need(targets, "targets", dtype=torch.int32, shape=(N,))
    _need(mask, "mask", dtype=torch.uint8, shape=(N,))
    return GhHead(N=N, D=D, V=V, dtype=_abi.GH_BF16 if H.dtype == _BF16 else _abi.GH_FP32, row_tile=row_tile,
                  H=H.data_ptr(), W=W.data_ptr(), targets=targets.data_ptr(), mask=mask.data_ptr())


def forward_workspace_bytes(head: GhHead) -> int:
    return int(_lib().grpo_head_forward_workspace_size(ctypes.byref(head)))


def backward_workspace_bytes(head: GhHead) -> int:
    return int(_lib().grpo_head_backward_workspace_size(ctypes.byref(head)))


def backward_shard_workspace_bytes(head: GhHead, V_total: int) -> int:
    return int(_lib().grpo_head_backward_shard_workspace_size(ctypes.byref(head), int(V_total)))


def new_status(dev) -> torch.Tensor:
    return torch.zeros(1, dtype=torch.int32, device=dev)


def raise_on_status(status: torch.Tensor, allow: int = 0) -> int:
    """Read the device status word (synchronises) and raise on any bit not in ``allow``."""
    word = int(status.item())
    if word & ~allow:
        raise _abi.GhError(f"device status {word:#x} ({_abi.describe_status(word)})")
    return word


@_nvtx
def grpo_head_forward(H, W, targets, mask, *, old_logp=None, ref_logp=None, adv=None, seq_id=None,
                      num_seqs: int = 0, eps_low: float = 0.2, eps_high: float = 0.2, beta: float = 0.0,
                      reduction: str = "token_mean", norm: float = 0.0, delta: float = 0.0,
                      ratio_level: str = "token", seq_totals: bool = False, clip_count: bool = False,
                      row_tile: int = 0, want_coef: bool = True, status: Optional[torch.Tensor] = None,
                      out: Optional[dict] = None, workspace: Optional[torch.Tensor] = None):
    """Selected-token log-probs and LSE; with ``old_logp`` given, also the GRPO
    loss (loss, policy_loss, kl) and coef = d loss / d logp.  ``delta`` > 0
    caps the unclipped ratio (two-sided clip); ``ratio_level="sequence"`` uses
    one ratio per sequence; ``seq_totals`` also returns the per-sequence totals
    (seq_policy, seq_kl, seq_count) for a data-parallel reduction;
    ``clip_count`` returns ``num_clipped`` (int32 [1]), the active tokens whose
    policy gradient the clip cuts off.

    ``workspace``: a caller-owned CUDA byte buffer of at least
    forward_workspace_bytes(head) bytes; by default the binding's shared,
    grow-only buffer is used.  The shared buffer serves one stream at a time:
    calls whose GPU work overlaps, e.g. on different streams, must each pass
    their own.  A call captured into a CUDA graph keeps the workspace address it was
    given, so pass your own buffer when capturing (the shared one may be
    replaced by a larger one later).

    Returns a dict with logp, lse, and (GRPO) coef, loss3, plus status."""
    head = make_head(H, W, targets, mask, row_tile)
    dev = H.device
    N = head.N
    out = {} if out is None else out
    logp = out.get("logp") if out.get("logp") is not None else torch.empty(N, dtype=_F32, device=dev)
    lse = out.get("lse") if out.get("lse") is not None else torch.empty(N, dtype=_F32, device=dev)
    st = new_status(dev) if status is None else status
    g = None
    coef = loss3 = None
    if old_logp is not None:
        _need(old_logp, "old_logp", _F32, (N,))
        if ref_logp is not None:
            _need(ref_logp, "ref_logp", _F32, (N,))
        _need(adv, "adv", _F32)
        _need(seq_id, "seq_id", torch.int32, (N,))
        num_seqs = int(num_seqs or adv.numel())
        totals = None
        if seq_totals:
            totals = (torch.empty(num_seqs, dtype=_F32, device=dev), torch.empty(num_seqs, dtype=_F32, device=dev),
                      torch.empty(num_seqs, dtype=torch.int32, device=dev))
            out.update(seq_policy=totals[0], seq_kl=totals[1], seq_count=totals[2])
        clipped = None
        if clip_count:
            clipped = out.get("num_clipped") if out.get("num_clipped") is not None else \
                torch.empty(1, dtype=torch.int32, device=dev)
            out.update(num_clipped=clipped)
        g = GhGrpo(old_logp=old_logp.data_ptr(), ref_logp=ref_logp.data_ptr() if ref_logp is not None else None,
                   adv=adv.data_ptr(), seq_id=seq_id.data_ptr(), num_seqs=num_seqs,
                   reduction=_abi.REDUCTIONS[reduction], eps_low=eps_low, eps_high=eps_high, beta=beta,
                   delta=float(delta), norm=float(norm), ratio_level=_abi.RATIO_LEVELS[ratio_level], reserved=0,
                   seq_policy=totals[0].data_ptr() if totals else None,
                   seq_kl=totals[1].data_ptr() if totals else None,
                   seq_count=totals[2].data_ptr() if totals else None,
                   num_clipped=clipped.data_ptr() if clipped is not None else None)
        if want_coef:
            coef = out.get("coef") if out.get("coef") is not None else torch.empty(N, dtype=_F32, device=dev)
        loss3 = out.get("loss3") if out.get("loss3") is not None else torch.empty(3, dtype=_F32, device=dev)
    nbytes = forward_workspace_bytes(head)
    ws = _caller_workspace(workspace, nbytes) if workspace is not None else WORKSPACE.get(dev, nbytes)
    code = _lib().grpo_head_forward(ctypes.byref(head), ctypes.byref(g) if g is not None else None, _ptr(logp),
                                    _ptr(lse), _ptr(coef), _ptr(loss3), _ptr(st), _ptr(ws), nbytes, _stream(dev))
    _abi.check(code, "grpo_head_forward")
    out.update(logp=logp, lse=lse, coef=coef, loss3=loss3, status=st)
    return out


def vocab_shard_bounds(V_total: int, num_shards: int):
    """[(start, length)] of each vocabulary shard: whole 256-column splits,
    the remainder spread over the first shards (host-only library call)."""
    lib = _lib()
    out = []
    for r in range(num_shards):
        st, ln = ctypes.c_int64(), ctypes.c_int64()
        _abi.check(lib.gh_vocab_shard_bounds(int(V_total), int(num_shards), r, ctypes.byref(st), ctypes.byref(ln)),
                   "gh_vocab_shard_bounds")
        out.append((int(st.value), int(ln.value)))
    return out


@_nvtx
def grpo_head_logprob_shard(H, W_shard, targets, mask, *, vocab_start: int, V_total: int, row_tile: int = 0,
                            status: Optional[torch.Tensor] = None):
    """One vocabulary shard's split partials (part_m, part_s [S_shard, N]) and
    the target logits of the rows whose target lies in the shard (zy [N])."""
    head = make_head(H, W_shard, targets, mask, row_tile)
    dev = H.device
    N = head.N
    splits = int(_lib().gh_vocab_splits(head.V))
    part_m = torch.empty(splits, N, dtype=_F32, device=dev)
    part_s = torch.empty(splits, N, dtype=_F32, device=dev)
    zy = torch.zeros(N, dtype=_F32, device=dev)
    st = new_status(dev) if status is None else status
    code = _lib().grpo_head_logprob_shard(ctypes.byref(head), int(vocab_start), int(V_total), _ptr(part_m),
                                          _ptr(part_s), _ptr(zy), _ptr(st), _stream(dev))
    _abi.check(code, "grpo_head_logprob_shard")
    return dict(part_m=part_m, part_s=part_s, zy=zy, status=st)


@_nvtx
def grpo_logprob_merge(part_m, part_s, zy, shard_starts, targets, mask, *, V_total: int,
                       status: Optional[torch.Tensor] = None):
    """logp, lse [N] from the gathered shard partials (concatenated in shard
    order) and the shards' zy rows [num_shards, N]; shard_starts has
    num_shards + 1 host integers."""
    S, N = part_m.shape
    if S != int(_lib().gh_vocab_splits(int(V_total))):
        raise ValueError(f"part_m has {S} split rows; a {V_total}-column vocabulary has "
                         f"{int(_lib().gh_vocab_splits(int(V_total)))}")
    _need(part_m, "part_m", _F32)
    _need(part_s, "part_s", _F32, (S, N))
    num_shards = len(shard_starts) - 1
    _need(zy, "zy", _F32, (num_shards, N))
    _need(targets, "targets", torch.int32, (N,))
    _need(mask, "mask", torch.uint8, (N,))
    dev = part_m.device
    logp = torch.empty(N, dtype=_F32, device=dev)
    lse = torch.empty(N, dtype=_F32, device=dev)
    st = new_status(dev) if status is None else status
    starts = (ctypes.c_int64 * (num_shards + 1))(*[int(x) for x in shard_starts])
    code = _lib().grpo_logprob_merge(N, int(V_total), num_shards, starts, _ptr(part_m), _ptr(part_s), _ptr(zy),
                                     _ptr(targets), _ptr(mask), _ptr(logp), _ptr(lse), _ptr(st), _stream(dev))
    _abi.check(code, "grpo_logprob_merge")
    return dict(logp=logp, lse=lse, status=st)


@_nvtx
def grpo_head_backward_shard(H, W_shard, targets, mask, lse, coef, *, vocab_start: int, V_total: int,
                             grad_out=None, dW=None, accumulate_dW: bool = False, row_tile: int = 0,
                             status: Optional[torch.Tensor] = None):
    """One vocabulary shard's backward: dW for the shard's rows and the fp32
    dH partial G_shard W_shard (sum the shards' partials with grpo_dh_merge)."""
    head = make_head(H, W_shard, targets, mask, row_tile)
    dev = H.device
    N, D, V = head.N, head.D, head.V
    _need(lse, "lse", _F32, (N,))
    _need(coef, "coef", _F32, (N,))
    dHp = torch.empty(N, D, dtype=_F32, device=dev)
    if dW is None:
        if accumulate_dW:
            raise ValueError("accumulate_dW needs an existing dW")
        dW = torch.empty(V, D, dtype=_F32, device=dev)
    else:
        _need(dW, "dW", _F32, (V, D))
    st = new_status(dev) if status is None else status
    nbytes = backward_shard_workspace_bytes(head, V_total)
    ws = WORKSPACE.get(dev, nbytes)
    code = _lib().grpo_head_backward_shard(ctypes.byref(head), int(vocab_start), int(V_total), _ptr(lse), _ptr(coef),
                                           _ptr(grad_out), _ptr(dHp), _ptr(dW), 1 if accumulate_dW else 0, _ptr(st),
                                           _ptr(ws), nbytes, _stream(dev))
    _abi.check(code, "grpo_head_backward_shard")
    return dict(dH_partial=dHp, dW=dW, status=st)


@_nvtx
def grpo_dh_merge(dH_partials, dtype=torch.bfloat16, status: Optional[torch.Tensor] = None):
    """dH = sum over shards (in order) of the gathered fp32 partials [P, N, D]."""
    P, N, D = dH_partials.shape
    _need(dH_partials, "dH_partials", _F32)
    dev = dH_partials.device
    dH = torch.empty(N, D, dtype=dtype, device=dev)
    st = new_status(dev) if status is None else status
    code = _lib().grpo_dh_merge(P, N, D, _abi.GH_BF16 if dtype == _BF16 else _abi.GH_FP32, _ptr(dH_partials),
                                _ptr(dH), _ptr(st), _stream(dev))
    _abi.check(code, "grpo_dh_merge")
    return dH


@_nvtx
def grpo_loss_from_sequence_totals(seq_policy, seq_kl, seq_count, *, reduction: str = "token_mean",
                                   norm: float = 0.0, beta: float = 0.0, status: Optional[torch.Tensor] = None):
    """(loss, policy_loss, kl) from per-sequence totals gathered in global
    sequence order (bitwise equal to a single forward over the whole batch)."""
    S = seq_policy.numel()
    _need(seq_policy, "seq_policy", _F32, (S,))
    _need(seq_kl, "seq_kl", _F32, (S,))
    _need(seq_count, "seq_count", torch.int32, (S,))
    dev = seq_policy.device
    loss3 = torch.empty(3, dtype=_F32, device=dev)
    st = new_status(dev) if status is None else status
    code = _lib().grpo_loss_from_sequence_totals(S, _ptr(seq_policy), _ptr(seq_kl), _ptr(seq_count),
                                                 _abi.REDUCTIONS[reduction], float(norm), float(beta), _ptr(loss3),
                                                 _ptr(st), _stream(dev))
    _abi.check(code, "grpo_loss_from_sequence_totals")
    return dict(loss3=loss3, status=st)


@_nvtx
def gspo_segment_loss(logp, old_logp, mask, seg_id, num_segments: int, seg_adv, *, eps_low: float,
                      eps_high: float, divisor: float, token_weighted: bool = False, ref_logp=None,
                      beta: float = 0.0, status: Optional[torch.Tensor] = None,
                      workspace: Optional[torch.Tensor] = None):
    """GSPO sequence-level loss over packed documents (optionally with a
    per-segment mean k3 KL weighted by beta); returns loss [1], seg_ratio [S],
    coef [N], mean_logp [1], num_clipped [1] (live segments whose policy
    gradient the clip cuts off) and status.  ``workspace``: a caller-owned
    CUDA byte buffer of gspo_segment_workspace_size(num_segments) bytes; by
    default a fixed per-device buffer."""
    N = logp.numel()
    _need(logp, "logp", _F32, (N,))
    _need(old_logp, "old_logp", _F32, (N,))
    if ref_logp is not None:
        _need(ref_logp, "ref_logp", _F32, (N,))
    _need(mask, "mask", torch.uint8, (N,))
    _need(seg_id, "seg_id", torch.int32, (N,))
    _need(seg_adv, "seg_adv", _F32, (num_segments,))
    dev = logp.device
    loss = torch.empty(1, dtype=_F32, device=dev)
    ratio = torch.empty(num_segments, dtype=_F32, device=dev)
    coef = torch.empty(N, dtype=_F32, device=dev)
    mean_logp = torch.empty(1, dtype=_F32, device=dev)
    clipped = torch.empty(1, dtype=torch.int32, device=dev)
    st = new_status(dev) if status is None else status
    ws, nbytes = _seam_ws(dev, num_segments, workspace)
    code = _lib().gspo_segment_loss(N, _ptr(logp), _ptr(old_logp), _ptr(ref_logp), _ptr(mask), _ptr(seg_id),
                                    num_segments, _ptr(seg_adv), eps_low, eps_high, float(beta), float(divisor),
                                    1 if token_weighted else 0, _ptr(loss), _ptr(ratio), _ptr(coef), _ptr(mean_logp),
                                    _ptr(clipped), _ptr(st), _ptr(ws), nbytes, _stream(dev))
    _abi.check(code, "gspo_segment_loss")
    return dict(loss=loss, seg_ratio=ratio, coef=coef, mean_logp=mean_logp, num_clipped=clipped, status=st)


@_nvtx
def gspo_segment_partials(logp, old_logp, mask, seg_id, num_segments: int, *, ref_logp=None,
                          status: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None):
    """One sequence-parallel rank's GSPO partials: fsum [2S + 1], cnt [S + 1]."""
    N = logp.numel()
    _need(logp, "logp", _F32, (N,))
    _need(old_logp, "old_logp", _F32, (N,))
    _need(mask, "mask", torch.uint8, (N,))
    _need(seg_id, "seg_id", torch.int32, (N,))
    dev = logp.device
    fsum = torch.empty(2 * num_segments + 1, dtype=_F32, device=dev)
    cnt = torch.empty(num_segments + 1, dtype=torch.int32, device=dev)
    st = new_status(dev) if status is None else status
    ws, nbytes = _seam_ws(dev, num_segments, workspace)
    code = _lib().gspo_segment_partials(N, _ptr(logp), _ptr(old_logp), _ptr(ref_logp), _ptr(mask), _ptr(seg_id),
                                        num_segments, _ptr(fsum), _ptr(cnt), _ptr(st), _ptr(ws), nbytes,
                                        _stream(dev))
    _abi.check(code, "gspo_segment_partials")
    return dict(fsum=fsum, cnt=cnt, status=st)


@_nvtx
def gspo_segment_loss_from_partials(logp, mask, seg_id, num_segments: int, fsum_all, cnt_all, seg_adv, *,
                                    eps_low: float, eps_high: float, divisor: float, token_weighted: bool = False,
                                    ref_logp=None, beta: float = 0.0, status: Optional[torch.Tensor] = None,
                                    workspace: Optional[torch.Tensor] = None):
    """GSPO loss from the ranks' gathered partials ([R, 2S + 1], [R, S + 1]);
    coef for this rank's tokens."""
    N = logp.numel()
    R = fsum_all.shape[0]
    _need(logp, "logp", _F32, (N,))
    _need(mask, "mask", torch.uint8, (N,))
    _need(seg_id, "seg_id", torch.int32, (N,))
    _need(fsum_all, "fsum_all", _F32, (R, 2 * num_segments + 1))
    _need(cnt_all, "cnt_all", torch.int32, (R, num_segments + 1))
    _need(seg_adv, "seg_adv", _F32, (num_segments,))
    if ref_logp is not None:
        _need(ref_logp, "ref_logp", _F32, (N,))
    dev = logp.device
    loss = torch.empty(1, dtype=_F32, device=dev)
    ratio = torch.empty(num_segments, dtype=_F32, device=dev)
    coef = torch.empty(N, dtype=_F32, device=dev)
    mean_logp = torch.empty(1, dtype=_F32, device=dev)
    clipped = torch.empty(1, dtype=torch.int32, device=dev)
    st = new_status(dev) if status is None else status
    ws, nbytes = _seam_ws(dev, num_segments, workspace)
    code = _lib().gspo_segment_loss_from_partials(N, _ptr(logp), _ptr(ref_logp), _ptr(mask), _ptr(seg_id),
                                                  num_segments, R, _ptr(fsum_all), _ptr(cnt_all), _ptr(seg_adv),
                                                  eps_low, eps_high, float(beta), float(divisor),
                                                  1 if token_weighted else 0, _ptr(loss), _ptr(ratio), _ptr(coef),
                                                  _ptr(mean_logp), _ptr(clipped), _ptr(st), _ptr(ws), nbytes,
                                                  _stream(dev))
    _abi.check(code, "gspo_segment_loss_from_partials")
    return dict(loss=loss, seg_ratio=ratio, coef=coef, mean_logp=mean_logp, num_clipped=clipped, status=st)


@_nvtx
def grpo_head_backward(H, W, targets, mask, lse, coef, *, grad_out=None, dH=None, dW=None,
                       accumulate_dW: bool = False, row_tile: int = 0, status: Optional[torch.Tensor] = None,
                       workspace: Optional[torch.Tensor] = None):
    """dH [N, D] (dtype of H) and dW [V, D] fp32 from each row's LSE and coef.

    ``workspace``: a caller-owned CUDA byte buffer of at least
    backward_workspace_bytes(head) bytes; by default the binding's shared,
    grow-only buffer is used, which serves one stream at a time: calls whose
    GPU work overlaps, e.g. on different streams, must each pass their own."""
    head = make_head(H, W, targets, mask, row_tile)
    dev = H.device
    N, D, V = head.N, head.D, head.V
    _need(lse, "lse", _F32, (N,))
    _need(coef, "coef", _F32, (N,))
    if grad_out is not None:
        _need(grad_out, "grad_out", _F32)
    if dH is None:
        dH = torch.empty(N, D, dtype=H.dtype, device=dev)
    else:
        _need(dH, "dH", H.dtype, (N, D))
    if dW is None:
        if accumulate_dW:
            raise ValueError("accumulate_dW needs an existing dW")
        dW = torch.empty(V, D, dtype=_F32, device=dev)
    else:
        _need(dW, "dW", _F32, (V, D))
    st = new_status(dev) if status is None else status
    nbytes = backward_workspace_bytes(head)
    ws = _caller_workspace(workspace, nbytes) if workspace is not None else WORKSPACE.get(dev, nbytes)
    code = _lib().grpo_head_backward(ctypes.byref(head), _ptr(lse), _ptr(coef), _ptr(grad_out), _ptr(dH), _ptr(dW),
                                     1 if accumulate_dW else 0, _ptr(st), _ptr(ws), nbytes, _stream(dev))
    _abi.check(code, "grpo_head_backward")
    return dict(dH=dH, dW=dW, status=st)


@_nvtx
def grpo_group_advantage(rewards, group_size: int, eps: float = 1e-4, status: Optional[torch.Tensor] = None):
    """Group-normalised advantages of per-sequence rewards."""
    _need(rewards, "rewards", _F32)
    n = rewards.numel()
    dev = rewards.device
    adv = torch.empty(n, dtype=_F32, device=dev)
    st = new_status(dev) if status is None else status
    code = _lib().grpo_group_advantage(_ptr(rewards), n, int(group_size), float(eps), _ptr(adv), _ptr(st),
                                       _stream(dev))
    _abi.check(code, "grpo_group_advantage")
    return adv


def timeout_probe(timeout_ns: int, dev=None):
    """Run the bounded-wait self-test; returns the status word (synchronises)."""
    dev = torch.device("cuda") if dev is None else dev
    st = new_status(dev)
    _abi.check(_lib().gh_timeout_probe(_ptr(st), int(timeout_ns), _stream(dev)), "gh_timeout_probe")
    return int(st.item())


# ------------------------------------------------------------------ instrumentation
def profile_enable(on: bool = True):
    _lib().gh_profile_enable(1 if on else 0)


def profile_reset():
    _lib().gh_profile_reset()


def profile_read():
    """{kernel name: (launches, total_ms)} since the last reset (synchronises)."""
    lib = _lib()
    res = {}
    for k in range(_abi.NUM_KERNEL_KINDS):
        n = ctypes.c_int64()
        ms = ctypes.c_double()
        _abi.check(lib.gh_profile_read(k, ctypes.byref(n), ctypes.byref(ms)), "gh_profile_read")
        if n.value:
            res[lib.gh_kernel_kind_name(k).decode()] = (int(n.value), float(ms.value))
    return res


def launch_count() -> int:
    return int(_lib().gh_launch_count())
