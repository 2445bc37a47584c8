"""GPU parity of the GRPO variants against the fp64 oracle: the two-sided
clip cap (delta), one importance ratio per sequence, and the deterministic
data-parallel reduction (per-sequence totals gathered in sequence order give
the single-call loss bit for bit; advantage groups cut across ranks; dW
partials summed in rank order)."""
import numpy as np
import pytest
import torch

import oracle
from synth import CONFIGS, make_workload

from gpu_helpers import BF16_LOSS_REL, assert_grad_bf16, bf16_np, dev_head, dev_tensor, gpu_lib, host_head, loss_scale  # noqa: F401,E501

pytestmark = pytest.mark.gpu


def _prepare(old_noise, dtype=None):
    cfg = CONFIGS[2]
    w = make_workload(cfg, old_noise=old_noise, dtype=dtype)
    H, W = host_head(w)
    lp, _, _ = oracle.selected_logprob(H, W, w["targets"], w["mask"])
    w["old"] = (lp + w["u_old"]).astype(np.float32)
    w["ref"] = (lp + w["u_ref"]).astype(np.float32)
    w["adv"] = oracle.group_advantages(w["rewards"], w["group_size"]).astype(np.float32)
    return cfg, w, H, W


def _near_edges(o, w, edges, margin, seq_level):
    r = o["ratio"]
    near = np.zeros(r.shape, dtype=bool)
    for e in edges:
        near |= np.abs(r - e) < margin
    if seq_level:
        seq = w["seq_id"]
        near = np.array([near[seq == seq[i]].any() for i in range(len(r))])
    return near


@pytest.mark.parametrize("delta,ratio_level,old_noise", [
    (2.0, "token", 0.9),       # the cap binds on tokens with r > 2 and A < 0
    (1.1, "token", 0.5),       # a cap inside the clip band
    (0.0, "sequence", 0.5),
    (1.05, "sequence", 0.5),
])
@pytest.mark.parametrize("reduction,norm", [("token_mean", 0.0), ("seq_mean", 0.0), ("fixed", 1024.0)])
def test_variants_match_oracle(gpu_lib, delta, ratio_level, old_noise, reduction, norm):
    import gspo_logprob_gb300 as g
    cfg, w, H, W = _prepare(old_noise)
    o = oracle.forward_backward(H, W, w["targets"], w["mask"], w["seq_id"], w["adv"].astype(np.float64),
                                w["num_seqs"], w["old"].astype(np.float64), w["ref"].astype(np.float64), cfg.eps_low,
                                cfg.eps_high, cfg.beta, reduction, norm)
    o = dict(o)
    ores = oracle.grpo_loss(o["logp"], w["old"].astype(np.float64), w["ref"].astype(np.float64), w["mask"],
                            w["seq_id"], w["adv"].astype(np.float64), w["num_seqs"], cfg.eps_low, cfg.eps_high,
                            cfg.beta, reduction, norm, delta=delta, ratio_level=ratio_level)
    dH_o, dW_o = oracle.head_backward(H, W, w["targets"], o["lse"], ores["coef"])
    Hd, Wd, y, m = dev_head(w)
    fw = g.grpo_head_forward(Hd, Wd, y, m, old_logp=dev_tensor(w["old"]), ref_logp=dev_tensor(w["ref"]),
                             adv=dev_tensor(w["adv"]), seq_id=dev_tensor(w["seq_id"]), num_seqs=w["num_seqs"],
                             eps_low=cfg.eps_low, eps_high=cfg.eps_high, beta=cfg.beta, reduction=reduction,
                             norm=norm, delta=delta, ratio_level=ratio_level)
    bw = g.grpo_head_backward(Hd, Wd, y, m, fw["lse"], fw["coef"])
    torch.cuda.synchronize()
    assert int(fw["status"].item()) == 0
    if delta > 0 and ratio_level == "token" and delta > 1 + cfg.eps_high:
        # the cap must actually bind somewhere for the test to mean anything
        capped = (ores["ratio"] > delta) & (w["adv"][w["seq_id"]] < 0) & (w["mask"] > 0)
        assert capped.sum() >= 5
    loss = fw["loss3"].cpu().numpy().astype(np.float64)
    sc = loss_scale(ores)
    assert abs(loss[0] - ores["loss"]) <= BF16_LOSS_REL * sc, (loss[0], ores["loss"])
    assert abs(loss[1] - ores["policy"]) <= BF16_LOSS_REL * sc
    edges = [1 - cfg.eps_low, 1 + cfg.eps_high] + ([delta] if delta > 0 else [])
    far = ~_near_edges(ores, w, edges, 2e-4, ratio_level == "sequence")
    cg = fw["coef"].cpu().numpy()
    assert far.sum() > 100
    assert np.max(np.abs(cg[far] - ores["coef"][far])) <= 1e-3 * np.abs(ores["coef"]).max()
    if far.all():
        assert_grad_bf16(bf16_np(bw["dH"]), dH_o, "dH")
        assert_grad_bf16(bw["dW"].cpu().numpy(), dW_o, "dW")


@pytest.mark.parametrize("reduction,ratio_level", [("token_mean", "token"), ("seq_mean", "sequence"),
                                                   ("fixed", "token")])
def test_data_parallel_split_is_bitwise_identical(gpu_lib, reduction, ratio_level):
    # one call over the whole batch vs. two "ranks" that each own whole
    # sequences: each rank runs the forward on its tokens with the global
    # normaliser and returns per-sequence totals; the totals, gathered in
    # sequence order, reduce to the single call's (loss, policy, kl) bit for bit
    import gspo_logprob_gb300 as g
    cfg, w, H, W = _prepare(0.3)
    Hd, Wd, y, m = dev_head(w)
    S = w["num_seqs"]
    common = dict(eps_low=cfg.eps_low, eps_high=cfg.eps_high, beta=cfg.beta, reduction=reduction,
                  ratio_level=ratio_level, delta=2.0)
    norm_fixed = 1024.0
    whole = g.grpo_head_forward(Hd, Wd, y, m, old_logp=dev_tensor(w["old"]), ref_logp=dev_tensor(w["ref"]),
                                adv=dev_tensor(w["adv"]), seq_id=dev_tensor(w["seq_id"]), num_seqs=S,
                                norm=norm_fixed if reduction == "fixed" else 0.0, **common)
    mask = w["mask"]
    seq = w["seq_id"]
    counts = np.bincount(seq[mask > 0], minlength=S)
    norm = {"token_mean": float(counts.sum()), "seq_mean": float((counts > 0).sum()), "fixed": norm_fixed}[reduction]
    bounds = [(0, 3), (3, S)]   # contiguous sequence partition, uneven on purpose
    parts = []
    for s0, s1 in bounds:
        t0 = int(np.searchsorted(seq, s0, "left"))
        t1 = int(np.searchsorted(seq, s1, "left"))
        sl = slice(t0, t1)
        res = g.grpo_head_forward(Hd[sl].contiguous(), Wd, y[sl].contiguous(), m[sl].contiguous(),
                                  old_logp=dev_tensor(w["old"][sl]), ref_logp=dev_tensor(w["ref"][sl]),
                                  adv=dev_tensor(w["adv"][s0:s1]), seq_id=dev_tensor(seq[sl] - s0), num_seqs=s1 - s0,
                                  norm=norm, seq_totals=True, **common)
        parts.append((sl, res))
    gathered = [torch.cat([r[k] for _, r in parts]) for k in ("seq_policy", "seq_kl", "seq_count")]
    fin = g.grpo_loss_from_sequence_totals(*gathered, reduction=reduction, norm=norm, beta=cfg.beta)
    torch.cuda.synchronize()
    assert torch.equal(fin["loss3"].view(torch.int32), whole["loss3"].view(torch.int32))
    for sl, r in parts:
        assert torch.equal(r["coef"].view(torch.int32), whole["coef"][sl].view(torch.int32))
        assert torch.equal(r["logp"].view(torch.int32), whole["logp"][sl].view(torch.int32))


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_data_parallel_straddling_group_and_rank_ordered_dW(gpu_lib, dtype):
    # two "ranks" own whole sequences of one batch, cut inside an advantage
    # group (8 sequences, G = 8, cut after 3).  Each rank normalises advantages
    # from the gathered rewards of all sequences, runs forward + backward on its
    # tokens with the global normaliser and a fresh dW, and the dW partials are
    # summed in rank order.  Each rank's dH rows are bitwise the whole-batch dH
    # rows (a row's dH depends on neither the batch nor the row chunks, and the
    # fp32 GEMMs' K slices do not depend on the rows either); the rank-ordered
    # sum is the plain fp32 sum of the partials, the same bits on a repeat; and
    # dW matches the oracle over the whole batch.
    import gspo_logprob_gb300 as g
    from gpu_helpers import FP32_GRAD_ABS
    cfg, w, H, W = _prepare(0.05, dtype)    # ratios inside the clip band: no gradient switches at its edges
    Hd, Wd, y, m = dev_head(w)
    S, G = w["num_seqs"], w["group_size"]
    seq = w["seq_id"]
    rew = dev_tensor(w["rewards"])
    adv_all = g.grpo_group_advantage(rew, G)
    norm = float(w["mask"].sum())
    common = dict(eps_low=cfg.eps_low, eps_high=cfg.eps_high, beta=cfg.beta, norm=norm)
    whole_fw = g.grpo_head_forward(Hd, Wd, y, m, old_logp=dev_tensor(w["old"]), ref_logp=dev_tensor(w["ref"]),
                                   adv=adv_all, seq_id=dev_tensor(seq), num_seqs=S, **common)
    whole_bw = g.grpo_head_backward(Hd, Wd, y, m, whole_fw["lse"], whole_fw["coef"])
    pieces = []
    for s0, s1 in ((0, 3), (3, S)):
        t0, t1 = int(np.searchsorted(seq, s0, "left")), int(np.searchsorted(seq, s1, "left"))
        sl = slice(t0, t1)
        gathered = torch.cat([rew[:s0], rew[s0:s1], rew[s1:]])      # all-gather of the per-rank rewards
        adv = g.grpo_group_advantage(gathered, G)[s0:s1].contiguous()
        assert torch.equal(adv.view(torch.int32), adv_all[s0:s1].view(torch.int32))
        args = (Hd[sl].contiguous(), Wd, y[sl].contiguous(), m[sl].contiguous())
        fw = g.grpo_head_forward(*args, old_logp=dev_tensor(w["old"][sl]), ref_logp=dev_tensor(w["ref"][sl]),
                                 adv=adv, seq_id=dev_tensor(seq[sl] - s0), num_seqs=s1 - s0, **common)
        bw = g.grpo_head_backward(*args, fw["lse"], fw["coef"])
        pieces.append((sl, args, fw, bw))
    reduced = g.grpo_dh_merge(torch.stack([p[3]["dW"] for p in pieces]), dtype=torch.float32)
    again = g.grpo_dh_merge(torch.stack([p[3]["dW"] for p in pieces]), dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(reduced, pieces[0][3]["dW"] + pieces[1][3]["dW"])
    assert torch.equal(reduced.view(torch.int32), again.view(torch.int32))
    iv = torch.int16 if dtype == "bf16" else torch.int32
    for sl, _, fw, bw in pieces:
        assert torch.equal(fw["lse"].view(torch.int32), whole_fw["lse"][sl].view(torch.int32))
        assert torch.equal(bw["dH"].view(iv), whole_bw["dH"][sl].view(iv))
    o = oracle.forward_backward(H, W, w["targets"], w["mask"], seq, w["adv"].astype(np.float64), S,
                                w["old"].astype(np.float64), w["ref"].astype(np.float64), cfg.eps_low, cfg.eps_high,
                                cfg.beta, norm=norm)
    if dtype == "bf16":
        assert_grad_bf16(reduced.cpu().numpy(), o["dW"], "dW reduced over ranks")
    else:
        assert np.max(np.abs(reduced.cpu().numpy() - o["dW"])) <= FP32_GRAD_ABS
        assert np.max(np.abs(whole_bw["dH"].cpu().numpy() - o["dH"])) <= FP32_GRAD_ABS
