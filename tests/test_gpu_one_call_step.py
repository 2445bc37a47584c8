"""A whole 8B-vocabulary step in one call: 131072 tokens (128 sequences of
1024), D=4096, V=151936, passed to the forward and the backward at once,
against the same step as 16 micro-batch calls of 8192 tokens.

What the batch decomposition fixes: logp, LSE and coef of every row are the
same bits whatever the call holds (the vocabulary splits depend on V only,
and the normaliser is passed explicitly); the per-sequence totals of the one
call are the micro-batches' totals concatenated, and the loss of the one call
is the loss the data-parallel reduction gives from those totals; every dH row
is the same bits (a row's dH sums its own vocabulary blocks in a fixed
order).  dW sums over the rows: one call runs one MMA chain over all 131072
rows, the micro-batches sixteen chains added in order, so the two agree to
fp32 rounding only.  The inputs are drawn on the GPU from a seeded generator
(values of the 8B workload's distributions); the micro-batch path itself is
compared with the fp64 oracle in test_gpu_large_vocab_parity.py."""
import numpy as np
import pytest
import torch

from gpu_helpers import gpu_lib  # noqa: F401

pytestmark = pytest.mark.gpu

N_MB, MB, D, V, T = 16, 8192, 4096, 151936, 1024


def _inputs():
    gen = torch.Generator(device="cuda")
    gen.manual_seed(5150)
    N = N_MB * MB
    H = torch.randn(N, D, generator=gen, device="cuda").to(torch.bfloat16)
    W = (torch.randn(V, D, generator=gen, device="cuda") * 0.02).to(torch.bfloat16)
    y = torch.randint(0, V, (N,), generator=gen, device="cuda", dtype=torch.int32)
    rng = np.random.default_rng(5151)
    S = N // T
    lens = rng.integers(256, T + 1, S)
    mask = (np.arange(T)[None, :] < lens[:, None]).astype(np.uint8).reshape(-1)
    seq = np.repeat(np.arange(S, dtype=np.int32), T)
    adv = rng.standard_normal(S).astype(np.float32)
    m = torch.from_numpy(mask).cuda()
    return H, W, y, m, torch.from_numpy(seq).cuda(), torch.from_numpy(adv).cuda(), int(mask.sum())


def _bits(t):
    return t.contiguous().view(torch.int32 if t.dtype == torch.float32 else torch.int16)


def test_whole_step_in_one_call_equals_micro_batches(gpu_lib):
    import gspo_logprob_gb300 as g
    from gspo_logprob_gb300 import ops
    H, W, y, m, seq, adv, active = _inputs()
    N = H.shape[0]
    S = N // T
    spm = MB // T  # sequences per micro-batch

    # logp for the old/ref log-probs (the whole batch, no loss)
    ws_one = torch.empty(ops.forward_workspace_bytes(ops.make_head(H, W, y, m)), dtype=torch.uint8, device="cuda")
    base = g.grpo_head_forward(H, W, y, m, workspace=ws_one)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(5152)
    old = base["logp"] + (torch.rand(N, generator=gen, device="cuda") - 0.5) * 0.2
    ref = base["logp"] + (torch.rand(N, generator=gen, device="cuda") - 0.5) * 0.4
    loss_args = dict(eps_low=0.2, eps_high=0.28, beta=0.04, reduction="token_mean", norm=float(active),
                     seq_totals=True)

    one = g.grpo_head_forward(H, W, y, m, old_logp=old, ref_logp=ref, adv=adv, seq_id=seq, num_seqs=S,
                              workspace=ws_one, **loss_args)
    torch.cuda.synchronize()
    assert int(one["status"].item()) == 0
    assert torch.equal(_bits(one["logp"]), _bits(base["logp"]))

    ws_mb = torch.empty(ops.forward_workspace_bytes(ops.make_head(H[:MB], W, y[:MB], m[:MB])), dtype=torch.uint8,
                        device="cuda")
    parts = []
    for k in range(N_MB):
        r = slice(k * MB, (k + 1) * MB)
        s = slice(k * spm, (k + 1) * spm)
        parts.append(g.grpo_head_forward(H[r], W, y[r], m[r], old_logp=old[r], ref_logp=ref[r], adv=adv[s],
                                         seq_id=seq[r] - k * spm, num_seqs=spm, workspace=ws_mb, **loss_args))
        # the shared micro-batch workspace is reused by the next call on the same stream
    torch.cuda.synchronize()
    assert all(int(p["status"].item()) == 0 for p in parts)
    for key in ("logp", "lse", "coef", "seq_policy", "seq_kl", "seq_count"):
        cat = torch.cat([p[key] for p in parts])
        assert torch.equal(_bits(cat), _bits(one[key])), key
    totals = [torch.cat([p[k] for p in parts]) for k in ("seq_policy", "seq_kl", "seq_count")]
    dp = g.grpo_loss_from_sequence_totals(*totals, reduction="token_mean", norm=float(active), beta=0.04)
    torch.cuda.synchronize()
    assert torch.equal(_bits(dp["loss3"]), _bits(one["loss3"]))
    del ws_one, ws_mb

    # backward: one call over all rows, then the sixteen micro-batches
    head = ops.make_head(H, W, y, m)
    wsb = torch.empty(ops.backward_workspace_bytes(head), dtype=torch.uint8, device="cuda")
    assert wsb.numel() <= 0.75 * N * V * 2 + 4096
    bw = g.grpo_head_backward(H, W, y, m, one["lse"], one["coef"], workspace=wsb)
    torch.cuda.synchronize()
    assert int(bw["status"].item()) == 0
    del wsb
    wsb = torch.empty(ops.backward_workspace_bytes(ops.make_head(H[:MB], W, y[:MB], m[:MB])), dtype=torch.uint8,
                      device="cuda")
    dW = None
    dH_rows = []
    for k in range(N_MB):
        r = slice(k * MB, (k + 1) * MB)
        b = g.grpo_head_backward(H[r], W, y[r], m[r], one["lse"][r], one["coef"][r], dW=dW,
                                 accumulate_dW=dW is not None, workspace=wsb)
        dW = b["dW"]
        dH_rows.append(b["dH"])
        assert int(b["status"].item()) == 0
    torch.cuda.synchronize()
    assert torch.equal(_bits(torch.cat(dH_rows)), _bits(bw["dH"]))
    a, c = bw["dW"].double(), dW.double()
    assert torch.isfinite(a).all()
    scale = float(c.abs().max())
    assert scale > 0
    assert float((a - c).abs().max()) <= 1e-3 * scale
    cos = float((a * c).sum() / (a.norm() * c.norm()))
    assert cos >= 0.99999
