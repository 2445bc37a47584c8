"""CUDA-graph replay of the path.  Every library call only enqueues kernels and
asynchronous memsets on the caller's stream, on buffers the caller passes, so
a step of calls can be captured once and replayed.  Here a GRPO step
(advantage, forward + loss, backward over two vocabulary blocks) and a GSPO
step are captured with caller-owned workspaces, replayed on new inputs copied
into the captured buffers, and must give the bits an eager call gives."""
import math

import numpy as np
import pytest
import torch

from synth import CONFIGS, f32_to_bf16_bits, make_workload

from gpu_helpers import dev_tensor, gpu_lib  # noqa: F401

pytestmark = pytest.mark.gpu


def _capture(fn, warm=2):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(warm):
            fn()
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        res = fn()
    return graph, res


def _bits(t):
    return t.detach().clone().view(torch.uint8) if t.dtype != torch.bfloat16 else t.detach().clone().view(torch.int16)


def _grpo_inputs(micro_batch, V, D, rng_seed):
    cfg = CONFIGS[2]
    w = make_workload(cfg, micro_batch=micro_batch, N=768, with_weight=False)
    rng = np.random.default_rng(rng_seed)
    lp = -rng.uniform(0.5, 9.0, w["N"])
    old = (lp + w["u_old"]).astype(np.float32)
    ref = (lp + w["u_ref"]).astype(np.float32)
    return [dev_tensor(w["H"], "bf16"), dev_tensor(w["targets"]), dev_tensor(w["mask"]), dev_tensor(w["seq_id"]),
            dev_tensor(w["rewards"]), dev_tensor(old), dev_tensor(ref)], w


def test_graph_replay_matches_eager_grpo(gpu_lib):
    import gspo_logprob_gb300 as g
    from gspo_logprob_gb300 import ops
    cfg = CONFIGS[2]
    V, D = 20000, cfg.D                      # two backward vocabulary blocks (16384 + 3616 columns)
    rng = np.random.default_rng(7)
    W = dev_tensor(f32_to_bf16_bits((rng.standard_normal((V, D)) / math.sqrt(D)).astype(np.float32)), "bf16")
    A, wa = _grpo_inputs(0, V, D, 1)
    B, _ = _grpo_inputs(1, V, D, 2)
    N = A[0].shape[0]
    G, S = wa["group_size"], wa["num_seqs"]
    head = ops.make_head(A[0], W, A[1], A[2])
    ws_f = torch.empty(ops.forward_workspace_bytes(head), dtype=torch.uint8, device="cuda")
    ws_b = torch.empty(ops.backward_workspace_bytes(head), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dH = torch.empty(N, D, dtype=torch.bfloat16, device="cuda")
    dW = torch.empty(V, D, dtype=torch.float32, device="cuda")
    out = dict(logp=torch.empty(N, device="cuda"), lse=torch.empty(N, device="cuda"),
               coef=torch.empty(N, device="cuda"), loss3=torch.empty(3, device="cuda"))
    static = [torch.empty_like(x) for x in A]

    def step(bufs=static):
        H, y, m, seq, rew, old, ref = bufs
        adv = g.grpo_group_advantage(rew, G, status=status)
        fw = g.grpo_head_forward(H, W, y, m, old_logp=old, ref_logp=ref, adv=adv, seq_id=seq, num_seqs=S,
                                 eps_low=cfg.eps_low, eps_high=cfg.eps_high, beta=cfg.beta, status=status, out=out,
                                 workspace=ws_f)
        g.grpo_head_backward(H, W, y, m, fw["lse"], fw["coef"], dH=dH, dW=dW, status=status, workspace=ws_b)
        return [out["logp"], out["lse"], out["coef"], out["loss3"], dH, dW]

    eager = {}
    for name, inp in (("A", A), ("B", B)):
        res = step(inp)
        torch.cuda.synchronize()
        eager[name] = [_bits(t) for t in res]
    for s_, a_ in zip(static, A):
        s_.copy_(a_)
    graph, res = _capture(step)
    n_calls = ops.launch_count()
    for name, inp in (("A", A), ("B", B), ("A", A)):
        for s_, x in zip(static, inp):
            s_.copy_(x)
        graph.replay()
        torch.cuda.synchronize()
        for got, want in zip(res, eager[name]):
            assert torch.equal(_bits(got), want), name
    assert ops.launch_count() == n_calls      # replays run the captured kernels, no library calls
    assert int(status.item()) == 0


def test_graph_replay_matches_eager_gspo(gpu_lib):
    import gspo_logprob_gb300 as g
    from gspo_logprob_gb300 import ops
    cfg = CONFIGS[3]
    wa = make_workload(cfg, N=2048)
    wb = make_workload(cfg, micro_batch=1, N=2048, with_weight=False)
    W = dev_tensor(wa["W"], "bf16")
    S, G = cfg.num_docs, wa["group_size"]

    def inputs(w, seed):
        rng = np.random.default_rng(seed)
        old = (-rng.uniform(0.5, 9.0, w["N"]) + w["u_old"]).astype(np.float32)
        return [dev_tensor(w["H"], "bf16"), dev_tensor(w["targets"]), dev_tensor(w["mask"]), dev_tensor(w["seq_id"]),
                dev_tensor(w["rewards"]), dev_tensor(old)]

    A, B = inputs(wa, 3), inputs(wb, 4)
    N, D, V = 2048, cfg.D, cfg.V
    head = ops.make_head(A[0], W, A[1], A[2])
    ws_f = torch.empty(ops.forward_workspace_bytes(head), dtype=torch.uint8, device="cuda")
    ws_b = torch.empty(ops.backward_workspace_bytes(head), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dH = torch.empty(N, D, dtype=torch.bfloat16, device="cuda")
    dW = torch.empty(V, D, dtype=torch.float32, device="cuda")
    out = dict(logp=torch.empty(N, device="cuda"), lse=torch.empty(N, device="cuda"))
    static = [torch.empty_like(x) for x in A]

    def step(bufs=static):
        H, y, m, seg, rew, old = bufs
        adv = g.grpo_group_advantage(rew, G, status=status)
        fw = g.grpo_head_forward(H, W, y, m, status=status, out=out, workspace=ws_f)
        gs = g.gspo_segment_loss(fw["logp"], old, m, seg, S, adv, eps_low=cfg.eps_low, eps_high=cfg.eps_high,
                                 divisor=float(S), status=status)
        g.grpo_head_backward(H, W, y, m, fw["lse"], gs["coef"], dH=dH, dW=dW, status=status, workspace=ws_b)
        return [out["logp"], out["lse"], gs["loss"], gs["coef"], dH, dW]

    eager = {}
    for name, inp in (("A", A), ("B", B)):
        res = step(inp)
        torch.cuda.synchronize()
        eager[name] = [_bits(t) for t in res]
    for s_, a_ in zip(static, A):
        s_.copy_(a_)
    graph, res = _capture(step)
    for name, inp in (("B", B), ("A", A)):
        for s_, x in zip(static, inp):
            s_.copy_(x)
        graph.replay()
        torch.cuda.synchronize()
        for got, want in zip(res, eager[name]):
            assert torch.equal(_bits(got), want), name
    assert int(status.item()) == 0


def test_caller_workspace_is_checked(gpu_lib):
    import gspo_logprob_gb300 as g
    from gspo_logprob_gb300 import ops
    w = make_workload(CONFIGS[1], N=512, dtype="bf16")
    H, W = dev_tensor(w["H"], "bf16"), dev_tensor(w["W"], "bf16")
    y, m = dev_tensor(w["targets"]), dev_tensor(w["mask"])
    need = ops.forward_workspace_bytes(ops.make_head(H, W, y, m))
    with pytest.raises(ValueError, match="workspace"):
        g.grpo_head_forward(H, W, y, m, workspace=torch.empty(need - 1, dtype=torch.uint8, device="cuda"))
    with pytest.raises(ValueError, match="workspace"):
        g.grpo_head_forward(H, W, y, m, workspace=torch.empty(need, dtype=torch.uint8))
