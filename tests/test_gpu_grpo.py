"""GPU parity of the GRPO forward + backward (loss, coef, dH, dW) against the
fp64 oracle on the tiny fp32 and the small bf16 workloads, all three
reductions, both clip branches, advantages, determinism and error states."""
import numpy as np
import pytest
import torch

import oracle
from synth import CONFIGS, make_workload

from gpu_helpers import (BF16_LOSS_REL, FP32_GRAD_ABS, FP32_LOGP_ABS, FP32_LOSS_REL, assert_grad_bf16,  # noqa: F401
                         bf16_np, dev_head, dev_tensor, gpu_lib, host_head, loss_scale)

pytestmark = pytest.mark.gpu


def _prepare(cfg, dtype=None, old_noise=None, N=None):
    """Inputs of one call plus the oracle's logp-based old/ref log-probs."""
    w = make_workload(cfg, dtype=dtype, old_noise=old_noise, N=N)
    H, W = host_head(w)
    lp, lse, _ = oracle.selected_logprob(H, W, w["targets"], w["mask"])
    w["old"] = (lp + w["u_old"]).astype(np.float32)
    w["ref"] = (lp + w["u_ref"]).astype(np.float32)
    w["adv"] = oracle.group_advantages(w["rewards"], w["group_size"]).astype(np.float32)
    return w, H, W


def _gpu_step(w, reduction, norm, g0=None, row_tile=0):
    import gspo_logprob_gb300 as g
    Hd, Wd, y, m = dev_head(w)
    fw = g.grpo_head_forward(Hd, Wd, y, m, old_logp=dev_tensor(w["old"]), ref_logp=dev_tensor(w["ref"]),
                             adv=dev_tensor(w["adv"]), seq_id=dev_tensor(w["seq_id"]), num_seqs=w["num_seqs"],
                             eps_low=w["eps_low"], eps_high=w["eps_high"], beta=w["beta"], reduction=reduction,
                             norm=norm, row_tile=row_tile)
    go = None if g0 is None else torch.tensor([g0], dtype=torch.float32, device="cuda")
    bw = g.grpo_head_backward(Hd, Wd, y, m, fw["lse"], fw["coef"], grad_out=go, row_tile=row_tile)
    torch.cuda.synchronize()
    return fw, bw


def _oracle_step(w, H, W, reduction, norm, g0=1.0):
    # the oracle's loss is fed the oracle's own logp (old/ref are stored fp32 inputs)
    return oracle.forward_backward(H, W, w["targets"], w["mask"], w["seq_id"], w["adv"].astype(np.float64),
                                   w["num_seqs"], w["old"].astype(np.float64), w["ref"].astype(np.float64),
                                   w["eps_low"], w["eps_high"], w["beta"], reduction, norm, g0=g0)


def _near_clip(res, w, margin=1e-4):
    r = res["ratio"]
    return (np.abs(r - (1 - w["eps_low"])) < margin) | (np.abs(r - (1 + w["eps_high"])) < margin)


def test_config0_fp32_forward_backward(gpu_lib):
    w, H, W = _prepare(CONFIGS[0])
    fw, bw = _gpu_step(w, "token_mean", 0.0)
    o = _oracle_step(w, H, W, "token_mean", 0.0)
    assert int(fw["status"].item()) == 0 and int(bw["status"].item()) == 0
    assert not _near_clip(o, w).any()
    lp = fw["logp"].cpu().numpy()
    m = w["mask"] > 0
    assert np.max(np.abs(lp - o["logp"])) <= FP32_LOGP_ABS
    assert np.max(np.abs(fw["lse"].cpu().numpy() - o["lse"])) <= FP32_LOGP_ABS
    loss = fw["loss3"].cpu().numpy().astype(np.float64)
    assert abs(loss[0] - o["loss"]) <= FP32_LOSS_REL * loss_scale(o), (loss, o["loss"])
    assert abs(loss[1] - o["policy"]) <= FP32_LOSS_REL * loss_scale(o)
    assert abs(loss[2] - o["kl"]) <= FP32_LOSS_REL * max(abs(o["kl"]), 1e-12)
    assert np.max(np.abs(fw["coef"].cpu().numpy() - o["coef"])) <= 1e-6 * max(1.0, np.abs(o["coef"]).max())
    dH = bw["dH"].cpu().numpy()
    dW = bw["dW"].cpu().numpy()
    eh, ew = np.max(np.abs(dH - o["dH"])), np.max(np.abs(dW - o["dW"]))
    print(f"fp32 dH err {eh:.2e} dW err {ew:.2e}")
    assert eh <= FP32_GRAD_ABS and ew <= FP32_GRAD_ABS
    assert np.all(dH[~m] == 0.0)


@pytest.mark.parametrize("reduction,norm", [("token_mean", 0.0), ("seq_mean", 0.0), ("fixed", 1024.0)])
def test_config2_bf16_forward_backward(gpu_lib, reduction, norm):
    w, H, W = _prepare(CONFIGS[2])
    fw, bw = _gpu_step(w, reduction, norm)
    o = _oracle_step(w, H, W, reduction, norm)
    assert int(fw["status"].item()) == 0 and int(bw["status"].item()) == 0
    assert np.max(np.abs(fw["logp"].cpu().numpy() - o["logp"])) <= 3e-2
    loss = fw["loss3"].cpu().numpy().astype(np.float64)
    sc = loss_scale(o)
    assert abs(loss[0] - o["loss"]) <= BF16_LOSS_REL * sc, (loss[0], o["loss"], sc)
    assert abs(loss[1] - o["policy"]) <= BF16_LOSS_REL * sc
    far = ~_near_clip(o, w)
    cg = fw["coef"].cpu().numpy()
    assert np.max(np.abs(cg[far] - o["coef"][far])) <= 1e-3 * np.abs(o["coef"]).max()
    dH = bf16_np(bw["dH"])
    c1, r1 = assert_grad_bf16(dH, o["dH"], "dH")
    c2, r2 = assert_grad_bf16(bw["dW"].cpu().numpy(), o["dW"], "dW")
    print(f"{reduction}: dH cos {c1:.6f} rel {r1:.2e}; dW cos {c2:.6f} rel {r2:.2e}")


def test_config2_clip_branches(gpu_lib):
    # wider old-logp noise so both clip branches fire; gradients compared on
    # tokens away from the clip edges (exact ties are measure-zero)
    w, H, W = _prepare(CONFIGS[2], old_noise=0.5)
    fw, bw = _gpu_step(w, "token_mean", 0.0)
    o = _oracle_step(w, H, W, "token_mean", 0.0)
    m = w["mask"] > 0
    clipped = (o["act"] == 0) & m
    assert clipped.sum() > 20 and ((o["act"] == 1) & m).sum() > 20
    loss = fw["loss3"].cpu().numpy().astype(np.float64)
    assert abs(loss[0] - o["loss"]) <= BF16_LOSS_REL * loss_scale(o)
    far = ~_near_clip(o, w, 1e-3)
    cg = fw["coef"].cpu().numpy()
    # clipped tokens keep only the KL part of the coefficient; all tokens match the oracle
    assert np.max(np.abs(cg[far] - o["coef"][far])) <= 1e-3 * np.abs(o["coef"]).max()
    assert_grad_bf16(bf16_np(bw["dH"]), o["dH"], "dH")
    assert_grad_bf16(bw["dW"].cpu().numpy(), o["dW"], "dW")


def test_backward_deterministic_and_grad_output_scaling(gpu_lib):
    w, H, W = _prepare(CONFIGS[2])
    fw1, bw1 = _gpu_step(w, "token_mean", 0.0, g0=1.0)
    fw2, bw2 = _gpu_step(w, "token_mean", 0.0, g0=1.0)
    assert torch.equal(bw1["dH"].view(torch.int16), bw2["dH"].view(torch.int16))
    assert torch.equal(bw1["dW"].view(torch.int32), bw2["dW"].view(torch.int32))
    assert torch.equal(fw1["loss3"].view(torch.int32), fw2["loss3"].view(torch.int32))
    _, bw3 = _gpu_step(w, "token_mean", 0.0, g0=2.0)
    # scaling by 2 is exact in binary floating point
    assert torch.equal(bw3["dW"], 2.0 * bw1["dW"])
    assert torch.equal(bw3["dH"].float(), 2.0 * bw1["dH"].float())


def test_dW_accumulates_across_micro_batches(gpu_lib):
    import gspo_logprob_gb300 as g
    cfg = CONFIGS[2]
    w0, H0, W0 = _prepare(cfg)
    w1 = make_workload(cfg, micro_batch=1)
    lp1, _, _ = oracle.selected_logprob(*host_head(w1), w1["targets"], w1["mask"])
    w1["old"] = (lp1 + w1["u_old"]).astype(np.float32)
    w1["ref"] = (lp1 + w1["u_ref"]).astype(np.float32)
    w1["adv"] = oracle.group_advantages(w1["rewards"], w1["group_size"]).astype(np.float32)
    norm = float(w0["mask"].sum() + w1["mask"].sum())  # one normaliser for the whole step
    dW = None
    for k, w in enumerate((w0, w1)):
        Hd, Wd, y, m = dev_head(w)
        fw = g.grpo_head_forward(Hd, Wd, y, m, old_logp=dev_tensor(w["old"]), ref_logp=dev_tensor(w["ref"]),
                                 adv=dev_tensor(w["adv"]), seq_id=dev_tensor(w["seq_id"]), num_seqs=w["num_seqs"],
                                 eps_low=w["eps_low"], eps_high=w["eps_high"], beta=w["beta"], norm=norm)
        bw = g.grpo_head_backward(Hd, Wd, y, m, fw["lse"], fw["coef"], dW=dW, accumulate_dW=k > 0)
        dW = bw["dW"]
    o0 = _oracle_step(w0, H0, W0, "token_mean", norm)
    o1 = _oracle_step(w1, *host_head(w1), "token_mean", norm)
    assert_grad_bf16(dW.cpu().numpy(), o0["dW"] + o1["dW"], "dW accumulated")


def test_group_advantage_kernel(gpu_lib):
    import gspo_logprob_gb300 as g
    rng = np.random.default_rng(1)
    for G, n in ((4, 8), (8, 48), (1, 5), (8, 1024)):
        r = (rng.random(n) < 0.5).astype(np.float32)
        r[:G] = 1.0  # a group with identical rewards
        a = g.grpo_group_advantage(dev_tensor(r), G).cpu().numpy()
        np.testing.assert_allclose(a, oracle.group_advantages(r, G), rtol=1e-5, atol=1e-5)
        assert np.all(a[:G] == 0.0)


def test_no_active_tokens_and_bad_sequences(gpu_lib):
    import gspo_logprob_gb300 as g
    w, H, W = _prepare(CONFIGS[0])
    Hd, Wd, y, m = dev_head(w)
    z = torch.zeros_like(m)
    common = dict(old_logp=dev_tensor(w["old"]), ref_logp=dev_tensor(w["ref"]), adv=dev_tensor(w["adv"]),
                  num_seqs=w["num_seqs"], eps_low=0.2, eps_high=0.2, beta=0.04)
    fw = g.grpo_head_forward(Hd, Wd, y, z, seq_id=dev_tensor(w["seq_id"]), **common)
    assert int(fw["status"].item()) & 8  # GH_DEV_NO_ACTIVE
    assert torch.all(fw["loss3"] == 0) and torch.all(fw["coef"] == 0)
    fw = g.grpo_head_forward(Hd, Wd, y, z, seq_id=dev_tensor(w["seq_id"]), reduction="fixed", norm=64.0, **common)
    assert int(fw["status"].item()) == 0 and torch.all(fw["loss3"] == 0)
    bad = w["seq_id"].copy()
    bad[10], bad[11] = 3, 2  # decreasing
    fw = g.grpo_head_forward(Hd, Wd, y, m, seq_id=dev_tensor(bad), **common)
    assert int(fw["status"].item()) & 16  # GH_DEV_BAD_SEQ
