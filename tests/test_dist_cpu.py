"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2): each
rank gets disjoint micro-batches (and so different synthetic data), and the
step time reported is the maximum over ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mbs = bench.rank_micro_batches(rank, 3)
        t = bench.max_over_ranks(10.0 + rank, world, torch.device("cpu"))
        bench.barrier(world)
        q.put((rank, mbs, t))
    finally:
        dist.destroy_process_group()


def test_two_rank_sharding_and_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = {}
    try:
        for _ in range(2):
            r, mbs, t = q.get(timeout=120)
            out[r] = (mbs, t)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.terminate()
    assert set(out) == {0, 1}
    assert out[0][0] == [0, 1, 2] and out[1][0] == [3, 4, 5]   # disjoint micro-batches
    assert out[0][1] == 11.0 and out[1][1] == 11.0             # max over ranks


def test_rank_micro_batches_give_distinct_data():
    import bench
    from synth import CONFIGS, make_workload
    cfg = CONFIGS[2]
    a = make_workload(cfg, micro_batch=bench.rank_micro_batches(0, 1)[0], with_weight=False)
    b = make_workload(cfg, micro_batch=bench.rank_micro_batches(1, 1)[0], with_weight=False)
    assert not (a["H"] == b["H"]).all()


def _tp_worker(rank, world, port, q):
    # each CPU rank holds a vocabulary shard; it computes its fp64 per-split
    # (max, sumexp) partials, the ranks all-gather them in rank order and merge
    # them in global split order: the result is the whole-vocabulary LSE
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import numpy as np
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        V, D, N, SPLIT = 5000, 16, 24, 1024
        rng = np.random.default_rng(0)
        H = rng.standard_normal((N, D))
        W = rng.standard_normal((V, D)) * 0.5
        S = -(-V // SPLIT)
        base, extra = divmod(S, world)
        s0 = rank * base + min(rank, extra)
        ns = base + (1 if rank < extra else 0)
        c0, c1 = s0 * SPLIT, min(V, (s0 + ns) * SPLIT)
        Z = H @ W[c0:c1].T
        mine = []
        for a in range(c0, c1, SPLIT):
            blk = Z[:, a - c0:min(c1, a + SPLIT) - c0]
            mt = blk.max(axis=1)
            mine.append(np.stack([mt, np.exp(blk - mt[:, None]).sum(axis=1)]))
        mine = torch.tensor(np.stack(mine))                     # [ns, 2, N]
        sizes = [torch.zeros(1, dtype=torch.int64) for _ in range(world)]
        dist.all_gather(sizes, torch.tensor([mine.shape[0]]))
        width = max(int(x) for x in sizes)
        pad = torch.zeros(width, 2, N, dtype=torch.float64)
        pad[:mine.shape[0]] = mine
        got = [torch.zeros_like(pad) for _ in range(world)]
        dist.all_gather(got, pad)
        parts = torch.cat([got[r][:int(sizes[r])] for r in range(world)]).numpy()   # global split order
        m, s = np.full(N, -np.inf), np.zeros(N)
        for k in range(parts.shape[0]):
            mk, sk = parts[k, 0], parts[k, 1]
            M = np.maximum(m, mk)
            s = np.where(np.isfinite(m), s * np.exp(m - M), 0.0) + sk * np.exp(mk - M)
            m = M
        q.put((rank, (m + np.log(s)).tolist(), list(np.log(np.exp(H @ W.T).sum(axis=1)))))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_vocab_parallel_partials_exchange(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_tp_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = {}
    try:
        for _ in range(world):
            r, lse, ref = q.get(timeout=120)
            res[r] = (lse, ref)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.terminate()
    import numpy as np
    for r in range(world):
        np.testing.assert_allclose(res[r][0], res[r][1], rtol=0, atol=1e-12)
        assert res[r][0] == res[0][0]    # every rank merges to the same bits


def _dp_worker(rank, world, port, q):
    # each CPU rank owns whole sequences; per-sequence totals are gathered in
    # sequence order and summed there, and the global normaliser is an exact
    # integer all-reduce: the loss equals the single-rank loss bit for bit
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import numpy as np

    import oracle
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        rng = np.random.default_rng(5)
        nseq, T = 6, 12
        N = nseq * T
        logp = -rng.uniform(0.1, 4, N)
        old = logp + rng.uniform(-0.4, 0.4, N)
        ref = logp + rng.uniform(-0.2, 0.2, N)
        mask = (np.arange(T)[None, :] < rng.integers(2, T + 1, nseq)[:, None]).astype(np.uint8).reshape(-1)
        seq = np.repeat(np.arange(nseq), T)
        adv = rng.standard_normal(nseq)
        whole = oracle.grpo_loss(logp, old, ref, mask, seq, adv, nseq, 0.2, 0.28, 0.04)
        bounds = [(0, 2), (2, 5), (5, 6)][:world] if world == 3 else [(0, 4), (4, 6)]
        s0, s1 = bounds[rank]
        sl = slice(s0 * T, s1 * T)
        cnt = torch.tensor([int(mask[sl].sum())], dtype=torch.int64)
        dist.all_reduce(cnt)                                   # exact integer normaliser
        mine = oracle.grpo_loss(logp[sl], old[sl], ref[sl], mask[sl], seq[sl] - s0, adv[s0:s1], s1 - s0, 0.2, 0.28,
                                0.04, "token_mean", float(cnt.item()))
        tot = torch.zeros(nseq, dtype=torch.float64)
        tot[s0:s1] = torch.tensor(mine["per_seq_policy"])
        got = [torch.zeros(nseq, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(got, tot)
        per_seq = sum(got).numpy()                              # disjoint slices: exact
        policy = 0.0
        for s in range(nseq):                                   # sequence order, as the single rank sums
            policy += per_seq[s] * (1.0 / float(cnt.item()))
        q.put((rank, policy, whole["policy"], list(mine["coef"]), list(whole["coef"][sl])))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_data_parallel_sequence_totals_exchange(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_dp_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = {}
    try:
        for _ in range(world):
            r, pol, whole, coef, coef_whole = q.get(timeout=120)
            res[r] = (pol, whole, coef, coef_whole)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.terminate()
    for r in range(world):
        pol, whole, coef, coef_whole = res[r]
        assert pol == whole                                    # bitwise
        assert coef == coef_whole
