"""Oracle parity at the shape of the 8B-vocabulary GRPO workload (D=4096,
V=151936, bf16, beta=0.04, eps 0.2/0.28), gradients included.

Element-wise part: two 1024-token calls (the micro-batch's first two
sequences of 1024 tokens, one of each advantage sign) run forward, loss and
backward through the binding, the second adding its dW into the first's
(accumulate_dW) the way micro-batches of one step accumulate.  Both calls use
the normaliser of the two together (the cross-micro-batch token-mean
normaliser).  The oracle computes every output of both calls element by
element: logp, LSE, loss, coef, dH, and dW after each call (the second
against the sum of both calls' dW).  This covers every 16384-column
vocabulary block of the backward, the 4480-column tail block and the fp32
read-modify-write of dW.  With old = logp + U(-0.5, 0.5) both clip branches
fire for both advantage signs; tokens whose ratio would lie within 1e-4 of a
clip edge have their old log-prob moved 1e-3 away first (inputs drawn by the
oracle only), so no gradient decision sits on a rounding edge.

Full-size part: one whole 8192-token micro-batch, launched exactly as the
benchmark launches it.  The oracle computes every row's logp and LSE and so
every row's coef; dH is compared on sampled rows and dW on sampled vocabulary
rows (block edges, the tail block, target rows, random rows), each of which
the oracle forms from all 8192 tokens.  Accumulation, grad_output scaling and
run-to-run determinism are checked as exact properties.

Sources: Liger-Kernel PR #1160 "[GRPO] add chunked grpo streaming over
vocab", Testing Done (the correctness test compares the loss and the
gradients against a full reference); RL-Kernel PR #291 "[WS2][PR5][Logp] ...",
PR description (the 8B-scale vocabulary, fp32 logp and LSE)."""
import numpy as np
import pytest
import torch

import oracle
from synth import CONFIGS, make_workload

from gpu_helpers import (BF16_LOGP_ABS, BF16_LOSS_REL, assert_grad_bf16, bf16_np, dev_tensor,  # noqa: F401
                         gpu_lib)

pytestmark = pytest.mark.gpu

CFG = CONFIGS[4]   # one micro-batch: N=8192, D=4096, V=151936


@pytest.fixture(scope="module")
def mb0():
    """Micro-batch 0 of the 8B-vocabulary workload, with the exact fp64 view of W."""
    w = make_workload(CFG)
    w["W64"] = oracle.as_f64(w["W"], "bf16")
    w["W_dev"] = dev_tensor(w["W"], "bf16")
    return w


def _away_from_edges(lp, u_old, eps_low, eps_high):
    """old = lp + u with every ratio exp(-u) at least 1e-4 from a clip edge."""
    u = np.array(u_old, dtype=np.float64)
    for _ in range(4):
        r = np.exp(-u)
        near = (np.abs(r - (1 - eps_low)) < 1e-4) | (np.abs(r - (1 + eps_high)) < 1e-4)
        if not near.any():
            break
        u[near] += 1e-3
    return (lp + u).astype(np.float32), u


@pytest.mark.parametrize("old_noise", [CFG.old_noise, 0.5])
def test_two_sequence_calls_elementwise_with_dW_accumulation(gpu_lib, mb0, old_noise):
    import gspo_logprob_gb300 as g
    w = mb0
    T = CFG.seq_len
    A_all = oracle.group_advantages(w["rewards"], w["group_size"])
    assert A_all[0] < 0 < A_all[1]
    rng = np.random.default_rng(91)
    norm = float(w["mask"][:2 * T].sum())
    Wd = w["W_dev"]
    dW = None
    dW_sum_o = None
    for c in range(2):
        rows = slice(c * T, (c + 1) * T)
        H64 = oracle.as_f64(w["H"][rows], "bf16")
        y = w["targets"][rows]
        m = w["mask"][rows]
        seq = np.zeros(T, dtype=np.int32)
        adv = A_all[c:c + 1]
        lp_o, lse_o, _ = oracle.selected_logprob(H64, w["W64"], y, m)
        u_old = rng.uniform(-old_noise, old_noise, T)
        old, u_used = _away_from_edges(lp_o, u_old, CFG.eps_low, CFG.eps_high)
        ref = (lp_o + w["u_ref"][rows]).astype(np.float32)
        o = oracle.grpo_loss(lp_o, old.astype(np.float64), ref.astype(np.float64), m, seq, adv, 1, CFG.eps_low,
                             CFG.eps_high, CFG.beta, "token_mean", norm)
        if old_noise > 0.2:
            act = o["act"][m > 0]
            assert 0 < act.sum() < act.size, "the wide old-logp noise must clip some tokens and not others"
        dH_o, dW_o = oracle.head_backward(H64, w["W64"], y, lse_o, o["coef"])
        dW_sum_o = dW_o if dW_sum_o is None else dW_sum_o + dW_o
        del dW_o

        Hd = dev_tensor(w["H"][rows], "bf16")
        yd, md = dev_tensor(y), dev_tensor(m)
        fw = g.grpo_head_forward(Hd, Wd, yd, md, old_logp=dev_tensor(old), ref_logp=dev_tensor(ref),
                                 adv=dev_tensor(adv.astype(np.float32)), seq_id=dev_tensor(seq), num_seqs=1,
                                 eps_low=CFG.eps_low, eps_high=CFG.eps_high, beta=CFG.beta, norm=norm)
        bw = g.grpo_head_backward(Hd, Wd, yd, md, fw["lse"], fw["coef"], dW=dW, accumulate_dW=c > 0)
        torch.cuda.synchronize()
        assert int(fw["status"].item()) == 0 and int(bw["status"].item()) == 0
        dW = bw["dW"]
        lp = fw["logp"].cpu().numpy().astype(np.float64)
        lse = fw["lse"].cpu().numpy().astype(np.float64)
        assert np.max(np.abs(lse - lse_o)) <= BF16_LOGP_ABS
        assert np.max(np.abs(lp - lp_o)[m > 0]) <= BF16_LOGP_ABS
        loss3 = fw["loss3"].cpu().numpy().astype(np.float64)
        sc = max(abs(o["loss"]), o["abs_terms"])
        assert abs(loss3[0] - o["loss"]) <= BF16_LOSS_REL * sc
        assert abs(loss3[1] - o["policy"]) <= BF16_LOSS_REL * sc
        assert abs(loss3[2] - o["kl"]) <= BF16_LOSS_REL * max(abs(o["kl"]), 1e-30)
        coef = fw["coef"].cpu().numpy().astype(np.float64)
        np.testing.assert_allclose(coef, o["coef"], rtol=2e-3, atol=2e-3 * np.abs(o["coef"]).max())
        assert np.array_equal(coef != 0, o["coef"] != 0)          # exact: which tokens carry gradient
        assert_grad_bf16(bf16_np(bw["dH"]), dH_o, f"dH (call {c})")
        assert_grad_bf16(dW.cpu().numpy(), dW_sum_o, f"dW after call {c}" + (" (accumulated)" if c else ""))


def test_full_micro_batch_all_rows_and_sampled_dW_rows(gpu_lib, mb0):
    import gspo_logprob_gb300 as g
    w = mb0
    N, V = CFG.N, CFG.V
    H64 = oracle.as_f64(w["H"], "bf16")
    lp_o, lse_o, _ = oracle.selected_logprob(H64, w["W64"], w["targets"], w["mask"])
    old = (lp_o + w["u_old"]).astype(np.float32)
    ref = (lp_o + w["u_ref"]).astype(np.float32)
    adv = oracle.group_advantages(w["rewards"], w["group_size"])
    norm = float(w["mask"].sum())
    o = oracle.grpo_loss(lp_o, old.astype(np.float64), ref.astype(np.float64), w["mask"], w["seq_id"], adv,
                         w["num_seqs"], CFG.eps_low, CFG.eps_high, CFG.beta, "token_mean", norm)

    Hd = dev_tensor(w["H"], "bf16")
    Wd = w["W_dev"]
    y, m = dev_tensor(w["targets"]), dev_tensor(w["mask"])
    fw = g.grpo_head_forward(Hd, Wd, y, m, old_logp=dev_tensor(old), ref_logp=dev_tensor(ref),
                             adv=dev_tensor(adv.astype(np.float32)), seq_id=dev_tensor(w["seq_id"]),
                             num_seqs=w["num_seqs"], eps_low=CFG.eps_low, eps_high=CFG.eps_high, beta=CFG.beta,
                             norm=norm)
    bw = g.grpo_head_backward(Hd, Wd, y, m, fw["lse"], fw["coef"])
    torch.cuda.synchronize()
    assert int(fw["status"].item()) == 0 and int(bw["status"].item()) == 0
    act = w["mask"] > 0
    lp = fw["logp"].cpu().numpy().astype(np.float64)
    lse = fw["lse"].cpu().numpy().astype(np.float64)
    print(f"all rows: max |dlogp| {np.max(np.abs(lp - lp_o)[act]):.2e}  max |dlse| {np.max(np.abs(lse - lse_o)):.2e}")
    assert np.max(np.abs(lse - lse_o)) <= BF16_LOGP_ABS
    assert np.max(np.abs(lp - lp_o)[act]) <= BF16_LOGP_ABS
    loss3 = fw["loss3"].cpu().numpy().astype(np.float64)
    assert abs(loss3[0] - o["loss"]) <= BF16_LOSS_REL * max(abs(o["loss"]), o["abs_terms"])
    coef = fw["coef"].cpu().numpy().astype(np.float64)
    np.testing.assert_allclose(coef, o["coef"], rtol=2e-3, atol=2e-3 * np.abs(o["coef"]).max())

    # dH on sampled rows (first and last rows, every sequence represented)
    rng = np.random.default_rng(44)
    rows = np.unique(np.concatenate([[0, N - 1], rng.choice(np.flatnonzero(act), 30, replace=False)]))
    dH_rows_o, _ = oracle.head_backward(H64[rows], w["W64"], w["targets"][rows], lse_o[rows], o["coef"][rows])
    assert_grad_bf16(bf16_np(bw["dH"])[rows], dH_rows_o, "dH sampled rows")

    # dW on sampled vocabulary rows, each formed by the oracle from all N tokens:
    # tile and 16384-column block edges, the tail block, the last real row,
    # rows that are targets of active tokens, random rows
    targets_act = w["targets"][act]
    vs = np.unique(np.concatenate([
        [0, 255, 256, 16383, 16384, 147455, 147456, V - 1],
        rng.choice(targets_act, 12, replace=False),
        rng.choice(V, 12, replace=False)]))
    pos = {int(v): k for k, v in enumerate(vs)}
    y_sub = np.array([pos.get(int(t), -1) for t in w["targets"]], dtype=np.int64)
    _, dW_rows_o = oracle.head_backward(H64, w["W64"][vs], y_sub, lse_o, o["coef"])
    dW = bw["dW"]
    assert_grad_bf16(dW[torch.from_numpy(vs).cuda()].cpu().numpy(), dW_rows_o, "dW sampled vocabulary rows")

    # exact properties at full size: accumulation doubles, grad_output scales,
    # and a repeat gives the same bits
    dW_once = dW.clone()
    g.grpo_head_backward(Hd, Wd, y, m, fw["lse"], fw["coef"], dW=dW, accumulate_dW=True)
    assert torch.equal(dW, 2.0 * dW_once)
    go = torch.tensor([2.0], device="cuda")
    bw2 = g.grpo_head_backward(Hd, Wd, y, m, fw["lse"], fw["coef"], grad_out=go)
    assert torch.equal(bw2["dW"], 2.0 * dW_once)
    bw3 = g.grpo_head_backward(Hd, Wd, y, m, fw["lse"], fw["coef"])
    assert torch.equal(bw3["dW"].view(torch.int32), dW_once.view(torch.int32))
    assert torch.equal(bw3["dH"].view(torch.int16), bw["dH"].view(torch.int16))
