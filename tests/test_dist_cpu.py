"""Multi-rank logic on CPU ranks (gloo, world sizes 2 and 3).

The benchmark's host logic: each rank gets disjoint micro-batches (and so
different synthetic data), and the step time reported is the maximum over
ranks.  The exchanges a multi-rank trainer runs around the library, in the
library's own decomposition and layouts: vocabulary-parallel split partials
on the library's 256-column split grid (gh_vocab_shard_bounds,
gh_vocab_splits), gathered as [S_total, N] in shard order plus zy
[num_shards, N] (what grpo_logprob_merge reads); per-sequence loss totals
gathered in sequence order (what grpo_loss_from_sequence_totals reads); GSPO
segment partials gathered as [R, 2S + 1] and [R, S + 1] in rank order (what
gspo_segment_loss_from_partials reads)."""
import math
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


def _fold_splits(pm, ps):
    """fp64 fold of split partials [S, N] in the library merge's order: split
    groups g = k mod 8, each summed in increasing k, then the groups in order."""
    import numpy as np
    M = pm.max(axis=0)
    grp = []
    for g in range(8):
        acc = np.zeros(pm.shape[1])
        for k in range(g, pm.shape[0], 8):
            ok = np.isfinite(pm[k])
            acc = acc + np.where(ok, ps[k] * np.exp(np.where(ok, pm[k], 0.0) - M), 0.0)
        grp.append(acc)
    tot = grp[0]
    for g in range(1, 8):
        tot = tot + grp[g]
    return M + np.log(tot)


def _shard_partials(H, W_shard, y, c0):
    """One shard's per-split (max, sum exp) partials [S_shard, N] over its
    256-column splits and the target logits of rows whose target it owns."""
    import numpy as np
    Z = H @ W_shard.T
    N, ln = Z.shape
    pm, ps = [], []
    for a in range(0, ln, 256):
        blk = Z[:, a:a + 256]
        mt = blk.max(axis=1)
        pm.append(mt)
        ps.append(np.exp(blk - mt[:, None]).sum(axis=1))
    rel = y - c0
    own = (rel >= 0) & (rel < ln)
    zy = np.where(own, Z[np.arange(N), np.clip(rel, 0, ln - 1)], 0.0)
    return np.stack(pm), np.stack(ps), zy


def _tp_worker(rank, world, port, q):
    # each CPU rank holds the vocabulary shard the library's gh_vocab_shard_bounds
    # gives it (whole 256-column splits); it computes its fp64 split partials,
    # the ranks all-gather them into part_m / part_s [S_total, N] in shard order
    # and zy [num_shards, N] (the layout grpo_logprob_merge reads) and fold them
    # in the library's split order: every rank gets the same bits, and the bits
    # of the single-shard fold
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import numpy as np

    from gspo_logprob_gb300 import _abi, ops
    lib = _abi.load()
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        V, D, N = 5000, 16, 24
        rng = np.random.default_rng(0)
        H = rng.standard_normal((N, D))
        W = rng.standard_normal((V, D)) * 0.5
        y = rng.integers(0, V, N)
        bounds = ops.vocab_shard_bounds(V, world)
        c0, ln = bounds[rank]
        pm, ps, zy = _shard_partials(H, W[c0:c0 + ln], y, c0)
        assert pm.shape[0] == lib.gh_vocab_splits(ln)
        mine = torch.tensor(np.stack([pm, ps], axis=1))            # [S_shard, 2, N]
        sizes = [torch.zeros(1, dtype=torch.int64) for _ in range(world)]
        dist.all_gather(sizes, torch.tensor([mine.shape[0]]))
        width = max(int(x) for x in sizes)
        pad = torch.zeros(width, 2, N, dtype=torch.float64)
        pad[:mine.shape[0]] = mine
        got = [torch.zeros_like(pad) for _ in range(world)]
        dist.all_gather(got, pad)
        parts = torch.cat([got[r][:int(sizes[r])] for r in range(world)]).numpy()
        part_m, part_s = parts[:, 0], parts[:, 1]                  # [S_total, N], shard order = global split order
        zys = [torch.zeros(N, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(zys, torch.tensor(zy))
        zy_all = torch.stack(zys).numpy()                          # [num_shards, N]
        assert part_m.shape[0] == lib.gh_vocab_splits(V)
        starts = [b[0] for b in bounds] + [V]
        lse = _fold_splits(part_m, part_s)
        owner = np.searchsorted(np.array(starts[1:]), y, side="right")
        logp = zy_all[owner, np.arange(N)] - lse
        q.put((rank, lse.tolist(), logp.tolist()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_vocab_parallel_partials_exchange(world):
    import numpy as np

    from gspo_logprob_gb300 import build
    build()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_tp_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = {}
    try:
        for _ in range(world):
            r, lse, logp = q.get(timeout=120)
            res[r] = (lse, logp)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.terminate()
    # the single-shard fold of the same inputs (one rank holding all splits)
    V, D, N = 5000, 16, 24
    rng = np.random.default_rng(0)
    H = rng.standard_normal((N, D))
    W = rng.standard_normal((V, D)) * 0.5
    y = rng.integers(0, V, N)
    pm, ps, zy = _shard_partials(H, W, y, 0)
    lse1 = _fold_splits(pm, ps)
    from scipy.special import logsumexp
    np.testing.assert_allclose(lse1, logsumexp(H @ W.T, axis=1), rtol=0, atol=1e-12)
    for r in range(world):
        assert res[r][0] == lse1.tolist()                       # bitwise: any shard count, any rank
        assert res[r][1] == (zy - lse1).tolist()


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


def _sp_worker(rank, world, port, q):
    # GSPO under sequence parallelism: each CPU rank holds a contiguous piece of
    # the packed token sequence (documents span pieces) and forms the partials
    # gspo_segment_partials writes, fsum [2S + 1] = (S_s..., K_s..., sum m logp)
    # and cnt [S + 1] = (n_s..., sum m); the ranks all-gather them in rank order
    # into [R, 2S + 1] and [R, S + 1] (the layout gspo_segment_loss_from_partials
    # reads) and sum them over ranks in rank order
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import numpy as np

    from synth import CONFIGS, make_workload
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cfg = CONFIGS[3]
        w = make_workload(cfg, N=3000, masked_frac=0.1, with_weight=False)
        S = cfg.num_docs
        rng = np.random.default_rng(4)
        logp = -rng.uniform(0.05, 6.0, 3000)
        old = logp + w["u_old"]
        ref = logp + w["u_ref"]
        cuts = {2: [0, 1400, 3000], 3: [0, 777, 1901, 3000]}[world]
        a, b = cuts[rank], cuts[rank + 1]
        seg, m = w["seq_id"][a:b], w["mask"][a:b]
        fsum = np.zeros(2 * S + 1)
        cnt = np.zeros(S + 1, dtype=np.int64)
        for i in range(b - a):                                  # explicit loop over this piece's tokens
            s = int(seg[i])
            if s < 0 or not m[i]:
                continue
            d = ref[a + i] - logp[a + i]
            fsum[s] += logp[a + i] - old[a + i]
            fsum[S + s] += math.exp(d) - d - 1.0
            fsum[2 * S] += logp[a + i]
            cnt[s] += 1
            cnt[S] += 1
        fs = [torch.zeros(2 * S + 1, dtype=torch.float64) for _ in range(world)]
        cs = [torch.zeros(S + 1, dtype=torch.int64) for _ in range(world)]
        dist.all_gather(fs, torch.tensor(fsum))
        dist.all_gather(cs, torch.tensor(cnt))
        fsum_all = torch.stack(fs).numpy()                      # [R, 2S + 1], rank order
        cnt_all = torch.stack(cs).numpy()                       # [R, S + 1]
        Ssum = np.zeros(S)
        n = np.zeros(S, dtype=np.int64)
        for r in range(world):                                  # rank order
            Ssum = Ssum + fsum_all[r, :S]
            n = n + cnt_all[r, :S]
        lp_sum = sum(fsum_all[r, 2 * S] for r in range(world))
        act = int(sum(cnt_all[r, S] for r in range(world)))
        q.put((rank, n.tolist(), Ssum.tolist(), lp_sum / act))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_gspo_sequence_parallel_partials_exchange(world):
    import numpy as np

    import oracle
    from synth import CONFIGS, make_workload
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_sp_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = {}
    try:
        for _ in range(world):
            r, n, Ssum, mean_lp = q.get(timeout=120)
            res[r] = (n, Ssum, mean_lp)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.terminate()
    cfg = CONFIGS[3]
    w = make_workload(cfg, N=3000, masked_frac=0.1, with_weight=False)
    rng = np.random.default_rng(4)
    logp = -rng.uniform(0.05, 6.0, 3000)
    o = oracle.gspo_loss(logp, logp + w["u_old"], w["mask"], w["seq_id"], cfg.num_docs,
                         np.ones(cfg.num_docs), cfg.eps_low, cfg.eps_high, 1.0)
    for r in range(world):
        n, Ssum, mean_lp = res[r]
        assert res[r] == res[0]                                 # every rank: the same bits
        assert n == o["counts"].tolist()                        # exact counts
        live = np.array(n) > 0
        np.testing.assert_allclose(np.exp(np.array(Ssum)[live] / np.array(n)[live]), o["seg_ratio"][live],
                                   rtol=1e-12)
        assert abs(mean_lp - o["mean_logp"]) < 1e-12
    assert sum(1 for x in res[0][0] if x > 0) >= 5              # several documents, some cut across ranks
