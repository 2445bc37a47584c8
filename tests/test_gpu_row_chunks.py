"""The backward's row chunks (bf16): a vocabulary too narrow for any block
width to fit three quarters of N * V * 2 bytes per row makes the backward
walk the rows in chunks.  N = 1024, D = 512, V = 300: one 512-column block
takes 1024 bytes per row against a budget of 450, and two 256-column blocks
would need a 2048-byte fp32 dH accumulator row, so the rows go in chunks of
384 (384 + 384 + 256).  Checked: dH and dW against the fp64 oracle, dW
accumulated over two calls, and vocabulary shards (which chunk the rows as
the whole vocabulary does) giving dW rows bitwise equal to the whole
vocabulary's."""
import numpy as np
import pytest
import torch

import oracle
from synth import f32_to_bf16_bits

from gpu_helpers import assert_grad_bf16, bf16_np, dev_tensor, gpu_lib  # noqa: F401

pytestmark = pytest.mark.gpu

N, D, V = 1024, 512, 300


def _inputs(seed):
    rng = np.random.default_rng(seed)
    H = f32_to_bf16_bits(rng.standard_normal((N, D)).astype(np.float32))
    W = f32_to_bf16_bits((rng.standard_normal((V, D)) / np.sqrt(D)).astype(np.float32))
    y = rng.integers(0, V, N).astype(np.int32)
    m = (rng.random(N) < 0.8).astype(np.uint8)
    coef = (rng.standard_normal(N) * 1e-3).astype(np.float32) * m
    return H, W, y, m, coef


def test_workspace_takes_row_chunks(gpu_lib):
    import gspo_logprob_gb300 as g
    from gspo_logprob_gb300 import ops
    H, W, y, m, _ = _inputs(1)
    head = ops.make_head(dev_tensor(H, "bf16"), dev_tensor(W, "bf16"), dev_tensor(y), dev_tensor(m))
    # one 384-row chunk of the 512 padded columns, no accumulator, the tile counter
    assert ops.backward_workspace_bytes(head) == 384 * 512 * 2 + 256
    assert ops.backward_workspace_bytes(head) <= 0.75 * N * V * 2 + 256
    del g


def test_chunked_backward_matches_oracle_and_accumulates(gpu_lib):
    import gspo_logprob_gb300 as g
    dW = None
    dW_o = np.zeros((V, D))
    for seed in (2, 3):
        H, W, y, m, coef = _inputs(seed)
        W = _inputs(2)[1]                      # one head weight for both calls
        H64 = oracle.as_f64(H, "bf16")
        W64 = oracle.as_f64(W, "bf16")
        lp, lse_o, _ = oracle.selected_logprob(H64, W64, y, m)
        Hd, Wd, yd, md = dev_tensor(H, "bf16"), dev_tensor(W, "bf16"), dev_tensor(y), dev_tensor(m)
        fw = g.grpo_head_forward(Hd, Wd, yd, md)
        assert np.max(np.abs(fw["lse"].cpu().numpy() - lse_o)) < 3e-2
        bw = g.grpo_head_backward(Hd, Wd, yd, md, fw["lse"], dev_tensor(coef), dW=dW, accumulate_dW=dW is not None)
        torch.cuda.synchronize()
        assert int(fw["status"].item()) == 0 and int(bw["status"].item()) == 0
        dW = bw["dW"]
        dH_o, dW_c = oracle.head_backward(H64, W64, y, lse_o, coef.astype(np.float64))
        dW_o = dW_o + dW_c
        assert_grad_bf16(bf16_np(bw["dH"]), dH_o, f"dH (seed {seed})")
        assert_grad_bf16(dW.cpu().numpy(), dW_o, f"dW after seed {seed}")


def test_chunked_shards_give_the_whole_vocabulary_dW(gpu_lib):
    import gspo_logprob_gb300 as g
    H, W, y, m, coef = _inputs(4)
    Hd, Wd, yd, md = dev_tensor(H, "bf16"), dev_tensor(W, "bf16"), dev_tensor(y), dev_tensor(m)
    fw = g.grpo_head_forward(Hd, Wd, yd, md)
    cd = dev_tensor(coef)
    whole = g.grpo_head_backward(Hd, Wd, yd, md, fw["lse"], cd)
    parts = [g.grpo_head_backward_shard(Hd, Wd[s:s + n], yd, md, fw["lse"], cd, vocab_start=s, V_total=V)
             for s, n in g.vocab_shard_bounds(V, 2)]
    torch.cuda.synchronize()
    dW = torch.cat([p["dW"] for p in parts])
    assert torch.equal(dW.view(torch.int32), whole["dW"].view(torch.int32))
    dH = g.grpo_dh_merge(torch.stack([p["dH_partial"] for p in parts]))
    assert_grad_bf16(bf16_np(dH), bf16_np(whole["dH"]), "dH shards vs whole")
