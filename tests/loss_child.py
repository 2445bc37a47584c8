"""Child process of test_gpu_loss_kernels.py: runs the GRPO loss and the GSPO
seam over a set of cases under the environment it was started with (the
loss kernels' launch shape is a knob read once per process) and prints one
JSON object mapping each case to a digest of the bits of every output."""
import hashlib
import json
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

from synth import CONFIGS, make_workload  # noqa: E402

from gpu_helpers import dev_head, dev_tensor  # noqa: E402


def _digest(tensors):
    import torch
    h = hashlib.sha256()
    for t in tensors:
        h.update(t.detach().contiguous().cpu().view(torch.uint8).numpy().tobytes())
    return h.hexdigest()[:24]


def main():
    import torch

    import gspo_logprob_gb300 as g
    out = {}
    # GRPO on the small GRPO workload: reductions, ratio levels, the cap, and a
    # normaliser taken from the call (coef after the fold) or given (coef per sequence)
    cfg = CONFIGS[2]
    w = make_workload(cfg, old_noise=0.5)
    Hd, Wd, y, m = dev_head(w)
    base = g.grpo_head_forward(Hd, Wd, y, m)
    lp = base["logp"].cpu().numpy().astype(np.float64)
    old = dev_tensor((lp + w["u_old"]).astype(np.float32))
    ref = dev_tensor((lp + w["u_ref"]).astype(np.float32))
    adv = dev_tensor(np.linspace(-1.2, 0.9, w["num_seqs"]).astype(np.float32))
    seq = dev_tensor(w["seq_id"])
    for red, norm in (("token_mean", 0.0), ("token_mean", 700.0), ("seq_mean", 0.0), ("seq_mean", 8.0),
                      ("fixed", 1024.0)):
        for level in ("token", "sequence"):
            for delta in (0.0, 1.1):
                r = g.grpo_head_forward(Hd, Wd, y, m, old_logp=old, ref_logp=ref, adv=adv, seq_id=seq,
                                        num_seqs=w["num_seqs"], eps_low=cfg.eps_low, eps_high=cfg.eps_high,
                                        beta=cfg.beta, reduction=red, norm=norm, ratio_level=level, delta=delta,
                                        seq_totals=True, clip_count=True)
                torch.cuda.synchronize()
                assert int(r["status"].item()) == 0
                out[f"grpo/{red}/{norm}/{level}/{delta}"] = _digest(
                    [r[k] for k in ("loss3", "coef", "seq_policy", "seq_kl", "seq_count", "num_clipped")])
    # 8192 tokens (64 sequences of 128): more than the folding CTA writes coef
    # for, so a normaliser taken from the call uses the token-parallel coef kernel
    w = make_workload(cfg, N=8192, old_noise=0.5)
    Hd, Wd, y, m = dev_head(w)
    base = g.grpo_head_forward(Hd, Wd, y, m)
    lp = base["logp"].cpu().numpy().astype(np.float64)
    old = dev_tensor((lp + w["u_old"]).astype(np.float32))
    ref = dev_tensor((lp + w["u_ref"]).astype(np.float32))
    adv = dev_tensor(np.linspace(-1.2, 0.9, w["num_seqs"]).astype(np.float32))
    seq = dev_tensor(w["seq_id"])
    for red in ("token_mean", "seq_mean"):
        for level in ("token", "sequence"):
            r = g.grpo_head_forward(Hd, Wd, y, m, old_logp=old, ref_logp=ref, adv=adv, seq_id=seq,
                                    num_seqs=w["num_seqs"], eps_low=cfg.eps_low, eps_high=cfg.eps_high,
                                    beta=cfg.beta, reduction=red, ratio_level=level, seq_totals=True,
                                    clip_count=True)
            torch.cuda.synchronize()
            assert int(r["status"].item()) == 0
            out[f"grpo8192/{red}/{level}"] = _digest(
                [r[k] for k in ("loss3", "coef", "seq_policy", "seq_kl", "seq_count", "num_clipped")])
    # GSPO on the packed layout (masked tokens, the -1 tail), with the KL term,
    # and its sequence-parallel pair over three pieces
    cfg = CONFIGS[3]
    w = make_workload(cfg, masked_frac=0.1, with_weight=False, old_noise=0.01)
    rng = np.random.default_rng(7)
    N, S = cfg.N, cfg.num_docs
    logp = (-rng.uniform(0.05, 6.0, N)).astype(np.float32)
    oldg = (logp.astype(np.float64) + w["u_old"]).astype(np.float32)
    refg = (logp.astype(np.float64) + w["u_ref"]).astype(np.float32)
    A = dev_tensor(np.linspace(-1.0, 1.0, S).astype(np.float32))
    args = dict(eps_low=cfg.eps_low, eps_high=cfg.eps_high, divisor=float(S))
    for tw in (False, True):
        r = g.gspo_segment_loss(dev_tensor(logp), dev_tensor(oldg), dev_tensor(w["mask"]), dev_tensor(w["seq_id"]),
                                S, A, token_weighted=tw, ref_logp=dev_tensor(refg), beta=0.05, **args)
        torch.cuda.synchronize()
        assert int(r["status"].item()) == 0
        out[f"gspo/{tw}"] = _digest([r[k] for k in ("loss", "seg_ratio", "coef", "mean_logp", "num_clipped")])
    cuts = [0, 5000, 11111, N]
    parts = [g.gspo_segment_partials(dev_tensor(logp[a:b]), dev_tensor(oldg[a:b]), dev_tensor(w["mask"][a:b]),
                                     dev_tensor(w["seq_id"][a:b]), S, ref_logp=dev_tensor(refg[a:b]))
             for a, b in zip(cuts[:-1], cuts[1:])]
    fsum = torch.stack([p["fsum"] for p in parts])
    cnt = torch.stack([p["cnt"] for p in parts])
    for k, (a, b) in enumerate(zip(cuts[:-1], cuts[1:])):
        r = g.gspo_segment_loss_from_partials(dev_tensor(logp[a:b]), dev_tensor(w["mask"][a:b]),
                                              dev_tensor(w["seq_id"][a:b]), S, fsum, cnt, A,
                                              ref_logp=dev_tensor(refg[a:b]), beta=0.05, **args)
        torch.cuda.synchronize()
        out[f"gspo_sp/{k}"] = _digest([r[k2] for k2 in ("loss", "seg_ratio", "coef", "mean_logp", "num_clipped")])
    out["gspo_sp/partials"] = _digest([fsum, cnt])
    print(json.dumps(out))


if __name__ == "__main__":
    main()
