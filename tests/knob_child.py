"""Child process of test_gpu_knobs.py: runs one GRPO forward + backward under
the tuning environment it was started with (tile heights, raster groups,
vocabulary block width) and checks it against the fp64 oracle.  Exit code 0
on success (printing digests of the dW and dH bits); prints the errors."""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

import oracle  # noqa: E402
from synth import CONFIGS, make_workload  # noqa: E402

from gpu_helpers import assert_grad_bf16, bf16_np, dev_head, dev_tensor, host_head, loss_scale  # noqa: E402


def main(dtype):
    import torch

    import gspo_logprob_gb300 as g
    cfg = CONFIGS[2]
    # V=3000 with D=192, N=768: several 256-column tiles, a ragged last tile and,
    # with a small block width, several backward vocabulary blocks
    w = make_workload(cfg, dtype=dtype, N=768)
    rng = np.random.default_rng(11)
    V, D = 3000, 192
    Wf = (rng.standard_normal((V, D)) / np.sqrt(D)).astype(np.float32)
    Hf = rng.standard_normal((768, D)).astype(np.float32)
    from synth import f32_to_bf16_bits
    w["W"] = f32_to_bf16_bits(Wf) if dtype == "bf16" else Wf
    w["H"] = f32_to_bf16_bits(Hf) if dtype == "bf16" else Hf
    w["targets"] = rng.integers(0, V, 768).astype(np.int32)
    H, W = host_head(w)
    lp, lse, _ = oracle.selected_logprob(H, W, w["targets"], w["mask"])
    old = (lp + w["u_old"]).astype(np.float32)
    ref = (lp + w["u_ref"]).astype(np.float32)
    adv = oracle.group_advantages(w["rewards"], w["group_size"]).astype(np.float32)
    o = oracle.forward_backward(H, W, w["targets"], w["mask"], w["seq_id"], adv.astype(np.float64), w["num_seqs"],
                                old.astype(np.float64), ref.astype(np.float64), cfg.eps_low, cfg.eps_high, cfg.beta)
    Hd, Wd, y, m = dev_head(w)
    fw = g.grpo_head_forward(Hd, Wd, y, m, old_logp=dev_tensor(old), ref_logp=dev_tensor(ref), adv=dev_tensor(adv),
                             seq_id=dev_tensor(w["seq_id"]), num_seqs=w["num_seqs"], eps_low=cfg.eps_low,
                             eps_high=cfg.eps_high, beta=cfg.beta)
    bw = g.grpo_head_backward(Hd, Wd, y, m, fw["lse"], fw["coef"])
    torch.cuda.synchronize()
    assert int(fw["status"].item()) == 0 and int(bw["status"].item()) == 0
    e = float(np.max(np.abs(fw["logp"].cpu().numpy() - o["logp"])))
    assert e < (1e-4 if dtype == "fp32" else 1e-3), e
    assert abs(float(fw["loss3"][0].item()) - o["loss"]) <= 2e-3 * loss_scale(o)
    if dtype == "bf16":
        assert_grad_bf16(bf16_np(bw["dH"]), o["dH"], "dH")
        assert_grad_bf16(bw["dW"].cpu().numpy(), o["dW"], "dW")
    else:
        assert np.max(np.abs(bw["dH"].cpu().numpy() - o["dH"])) <= 2e-4
        assert np.max(np.abs(bw["dW"].cpu().numpy() - o["dW"])) <= 2e-4
    # the row tile (and with it the kernel variant) must not change a bit
    ref = g.grpo_head_forward(Hd, Wd, y, m, row_tile=128)
    for rt in (0, 64, 256):
        o2 = g.grpo_head_forward(Hd, Wd, y, m, row_tile=rt)
        assert torch.equal(o2["lse"].view(torch.int32), ref["lse"].view(torch.int32)), rt
        assert torch.equal(o2["logp"].view(torch.int32), ref["logp"].view(torch.int32)), rt
    import hashlib
    dig = lambda t: hashlib.sha256(t.contiguous().cpu().view(torch.uint8).numpy().tobytes()).hexdigest()[:16]
    print("ok", dtype, e, "dW=" + dig(bw["dW"]), "dH=" + dig(bw["dH"]), "lse=" + dig(fw["lse"]), "logp=" + dig(fw["logp"]))


if __name__ == "__main__":
    main(sys.argv[1])
