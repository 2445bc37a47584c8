"""Seeded workload definitions and raw-input draws (no method arithmetic).

Every draw comes from ``numpy.random.Generator`` (PCG64) seeded from
``SeedSequence(1000 + config index)``; independent streams (head weight,
each micro-batch, layout, rewards, noise) are spawned children of that seed
so that one micro-batch can be drawn without drawing the others.

The five workloads follow the test shapes the pages quote for the fused
GRPO head (Liger-Kernel PR #1160, "Testing Done" failure list: B=1, T=4096,
D=256, V=5000 and B=8, T=128, D=1024, V=4096), the 8B-scale vocabulary the
RL-Kernel PR #291 description targets (Qwen3-8B: D=4096, V=151936) and the
packed uneven documents of Fast-LLM PR #554 ("Correctness").  The pages name
no public dataset; all values are synthetic.
"""
from __future__ import annotations

import dataclasses
import os
from typing import Optional

import numpy as np


# --------------------------------------------------------------------------
# bf16 as raw bits (round to nearest, ties to even)
# --------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return uint16 bits.

    Inputs must be finite (all draws here are)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact float32 value of each bf16 bit pattern."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# --------------------------------------------------------------------------
# workload table
# --------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class WorkloadConfig:
    index: int
    name: str
    kind: str               # "grpo" | "logp" | "gspo"
    N: int                  # tokens per call (one micro-batch)
    D: int
    V: int
    dtype: str              # "fp32" | "bf16"
    w_std: Optional[float]  # None -> 1/sqrt(D)
    # GRPO padded layout: num_prompts x group_size sequences of seq_len tokens
    num_prompts: int = 0
    group_size: int = 0
    seq_len: int = 0
    len_lo: int = 0
    len_hi: int = 0
    micro_batches: int = 1  # calls per step (each call = N tokens)
    eps_low: float = 0.2
    eps_high: float = 0.2
    beta: float = 0.0
    reductions: tuple = ("token_mean",)
    old_noise: float = 0.1  # old_logp = logp + U(-old_noise, old_noise)
    ref_noise: float = 0.2  # ref_logp = logp + U(-ref_noise, ref_noise)
    # GSPO packed layout
    num_docs: int = 0
    doc_len_lo: int = 0
    doc_len_hi: int = 0

    @property
    def seed(self) -> int:
        return 1000 + self.index

    @property
    def num_seqs(self) -> int:
        """Sequences (GRPO) or documents (GSPO) in one call."""
        if self.kind == "gspo":
            return self.num_docs
        if self.kind == "grpo":
            return self.num_prompts * self.group_size // self.micro_batches
        return 0

    @property
    def total_tokens(self) -> int:
        return self.N * self.micro_batches

    def weight_std(self) -> float:
        return float(self.w_std) if self.w_std is not None else 1.0 / float(np.sqrt(self.D))


CONFIGS = (
    WorkloadConfig(
        index=0, name="tiny_fp32_grpo", kind="grpo", N=256, D=64, V=500, dtype="fp32",
        w_std=None, num_prompts=2, group_size=4, seq_len=32, len_lo=8, len_hi=32,
        eps_low=0.2, eps_high=0.2, beta=0.04, reductions=("token_mean",)),
    WorkloadConfig(
        index=1, name="selective_logp", kind="logp", N=4096, D=256, V=5000, dtype="bf16",
        w_std=None),
    WorkloadConfig(
        index=2, name="bf16_grpo_small", kind="grpo", N=1024, D=1024, V=4096, dtype="bf16",
        w_std=None, num_prompts=1, group_size=8, seq_len=128, len_lo=8, len_hi=128,
        eps_low=0.2, eps_high=0.28, beta=0.1,
        reductions=("token_mean", "seq_mean", "fixed")),
    WorkloadConfig(
        index=3, name="bf16_gspo_packed", kind="gspo", N=16384, D=2048, V=32000, dtype="bf16",
        w_std=None, group_size=8, num_docs=48, doc_len_lo=64, doc_len_hi=640,
        eps_low=3e-4, eps_high=4e-4, beta=0.0),
    WorkloadConfig(
        index=4, name="bf16_grpo_8b_vocab", kind="grpo", N=8192, D=4096, V=151936, dtype="bf16",
        w_std=0.02, num_prompts=16, group_size=8, seq_len=1024, len_lo=256, len_hi=1024,
        micro_batches=16, eps_low=0.2, eps_high=0.28, beta=0.04,
        reductions=("token_mean",)),
)


MAX_MICRO_BATCHES = 1024
CHUNK_ROWS = 2048


def _streams(seed: int):
    """Independent child seed sequences: head weight, layout, rewards, noise,
    then one per micro-batch."""
    return np.random.SeedSequence(seed).spawn(4 + MAX_MICRO_BATCHES)


def _gen(ss):
    return np.random.Generator(np.random.PCG64(ss))


def _normal_rows(ss, rows: int, cols: int, std: float) -> np.ndarray:
    """N(0, std^2) float32 [rows, cols]; row chunks of CHUNK_ROWS come from their
    own child streams and are drawn in parallel threads, so the values do not
    depend on the thread count."""
    out = np.empty((rows, cols), dtype=np.float32)
    nchunk = (rows + CHUNK_ROWS - 1) // CHUNK_ROWS
    kids = ss.spawn(nchunk)

    def fill(c):
        r0 = c * CHUNK_ROWS
        r1 = min(rows, r0 + CHUNK_ROWS)
        _gen(kids[c]).standard_normal((r1 - r0, cols), dtype=np.float32, out=out[r0:r1])
        if std != 1.0:
            out[r0:r1] *= np.float32(std)

    if nchunk == 1:
        fill(0)
    else:
        import concurrent.futures as cf
        with cf.ThreadPoolExecutor(max_workers=min(nchunk, os.cpu_count() or 1)) as ex:
            list(ex.map(fill, range(nchunk)))
    return out


def _bf16_rows(x: np.ndarray) -> np.ndarray:
    """f32_to_bf16_bits applied chunk-wise in parallel threads."""
    out = np.empty(x.shape, dtype=np.uint16)
    n = x.shape[0]
    if n <= CHUNK_ROWS:
        out[...] = f32_to_bf16_bits(x)
        return out
    import concurrent.futures as cf

    def conv(r0):
        out[r0:r0 + CHUNK_ROWS] = f32_to_bf16_bits(x[r0:r0 + CHUNK_ROWS])

    with cf.ThreadPoolExecutor(max_workers=os.cpu_count() or 1) as ex:
        list(ex.map(conv, range(0, n, CHUNK_ROWS)))
    return out


# --------------------------------------------------------------------------
# raw draws
# --------------------------------------------------------------------------
def draw_grpo_layout(rng, num_seqs: int, seq_len: int, len_lo: int, len_hi: int):
    """Padded GRPO layout: sequence s owns tokens [s*T, (s+1)*T); its first
    L_s ~ U[len_lo, len_hi] (inclusive) tokens are the active completion."""
    lengths = rng.integers(len_lo, len_hi + 1, size=num_seqs).astype(np.int32)
    pos = np.arange(seq_len, dtype=np.int32)
    mask = (pos[None, :] < lengths[:, None]).astype(np.uint8).reshape(-1)
    seq_id = np.repeat(np.arange(num_seqs, dtype=np.int32), seq_len)
    return mask, seq_id, lengths


def draw_gspo_layout(rng, N: int, num_docs: int, lo: int, hi: int, masked_frac: float = 0.0):
    """Packed documents: lengths ~ U[lo, hi] laid out in order and cut at N
    (the document that crosses N is truncated, later ones dropped).  If the
    documents do not fill N, the tail has seg_id = -1 and mask = 0.  With
    masked_frac > 0 that fraction of document tokens (Bernoulli) is masked."""
    lengths = rng.integers(lo, hi + 1, size=num_docs).astype(np.int64)
    seg_id = np.full(N, -1, dtype=np.int32)
    pos = 0
    for d in range(num_docs):
        if pos >= N:
            break
        end = min(N, pos + int(lengths[d]))
        seg_id[pos:end] = d
        pos = end
    mask = (seg_id >= 0).astype(np.uint8)
    if masked_frac > 0.0:
        drop = rng.random(N) < masked_frac
        mask[drop] = 0
    return mask, seg_id, lengths.astype(np.int32)


def draw_rewards(rng, n: int, p: float = 0.5):
    """Bernoulli(p) scalar rewards, one per sequence/document (float32 0/1)."""
    return (rng.random(n) < p).astype(np.float32)


def draw_noise(rng, n: int, half_width: float):
    """U(-half_width, half_width) in float64 (added to a log-prob by the caller)."""
    return rng.uniform(-half_width, half_width, size=n)


# --------------------------------------------------------------------------
# one call's worth of raw inputs
# --------------------------------------------------------------------------
def make_workload(cfg: WorkloadConfig, micro_batch: int = 0, *, N: Optional[int] = None,
                  dtype: Optional[str] = None, masked_frac: float = 0.0,
                  old_noise: Optional[float] = None, with_weight: bool = True):
    """Raw inputs of one call (one micro-batch) of workload ``cfg``.

    Returns a dict: H, W (float32 or bf16 bits), targets int32, mask uint8,
    seq_id int32, rewards float32 [num_seqs], u_old / u_ref float64 noise,
    and the scalars of the config.  ``N`` overrides the token count (the
    GRPO layout then keeps whole sequences), ``dtype`` the storage type.
    W does not depend on ``micro_batch`` or ``N``; ``with_weight=False``
    skips drawing it (the caller already holds it)."""
    if not 0 <= micro_batch < MAX_MICRO_BATCHES:
        raise ValueError("micro_batch out of range")
    st = _streams(cfg.seed)
    rng_layout, rng_rew, rng_noise = _gen(st[1]), _gen(st[2]), _gen(st[3])
    ss_mb = st[4 + micro_batch]
    ss_h, ss_y = ss_mb.spawn(2)
    dt = dtype or cfg.dtype
    n_tok = N if N is not None else cfg.N
    out = dict(cfg=cfg, N=n_tok, D=cfg.D, V=cfg.V, dtype=dt,
               eps_low=cfg.eps_low, eps_high=cfg.eps_high, beta=cfg.beta)

    if with_weight:
        W = _normal_rows(st[0], cfg.V, cfg.D, cfg.weight_std())
        out["W"] = _bf16_rows(W) if dt == "bf16" else W
        del W
    H = _normal_rows(ss_h, n_tok, cfg.D, 1.0)
    out["H"] = _bf16_rows(H) if dt == "bf16" else H
    out["targets"] = _gen(ss_y).integers(0, cfg.V, size=n_tok, dtype=np.int64).astype(np.int32)

    # the layout streams are advanced micro_batch times so each micro-batch differs
    if cfg.kind == "grpo":
        T = cfg.seq_len
        if n_tok % T != 0:
            raise ValueError("GRPO layout needs N to be a multiple of the sequence length")
        nseq = n_tok // T
        for _ in range(micro_batch):
            draw_grpo_layout(rng_layout, nseq, T, cfg.len_lo, cfg.len_hi)
            draw_rewards(rng_rew, nseq)
        mask, seq_id, lengths = draw_grpo_layout(rng_layout, nseq, T, cfg.len_lo, cfg.len_hi)
        out.update(mask=mask, seq_id=seq_id, lengths=lengths, num_seqs=nseq,
                   group_size=min(cfg.group_size, nseq), rewards=draw_rewards(rng_rew, nseq))
    elif cfg.kind == "gspo":
        for _ in range(micro_batch):
            draw_gspo_layout(rng_layout, n_tok, cfg.num_docs, cfg.doc_len_lo, cfg.doc_len_hi,
                             masked_frac)
            draw_rewards(rng_rew, cfg.num_docs)
        mask, seg_id, lengths = draw_gspo_layout(rng_layout, n_tok, cfg.num_docs,
                                                 cfg.doc_len_lo, cfg.doc_len_hi, masked_frac)
        out.update(mask=mask, seq_id=seg_id, lengths=lengths, num_seqs=cfg.num_docs,
                   group_size=cfg.group_size, rewards=draw_rewards(rng_rew, cfg.num_docs))
    else:  # selective logp: every token active, no loss inputs
        out.update(mask=np.ones(n_tok, dtype=np.uint8), seq_id=np.zeros(n_tok, dtype=np.int32),
                   lengths=np.array([n_tok], dtype=np.int32), num_seqs=1, group_size=1,
                   rewards=np.zeros(1, dtype=np.float32))

    for _ in range(micro_batch):
        draw_noise(rng_noise, n_tok, 1.0)
        draw_noise(rng_noise, n_tok, 1.0)
    on = cfg.old_noise if old_noise is None else old_noise
    out["u_old"] = draw_noise(rng_noise, n_tok, on)
    out["u_ref"] = draw_noise(rng_noise, n_tok, cfg.ref_noise)
    return out
