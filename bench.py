#!/usr/bin/env python
"""Benchmark of the fused LM-head GRPO loss, forward + backward, on one GB300.

Workload (one step): the 8B-scale large-vocabulary GRPO head -- 16 prompts x
G=8 completions x T=1024 tokens = 131072 tokens, processed as 16 micro-batches
of 8192 tokens (one group each), D=4096, V=151936, bf16 H/W, token-mean loss
with the step's global active-token normaliser, eps 0.2/0.28, beta 0.04, fp32
LSE/logp, bf16 dH, dW accumulated in fp32 over the micro-batches.  A step is,
per micro-batch: group advantages, forward (logits + online LSE + GRPO loss +
coef), backward (dlogits recompute, dH, dW).

Prints ONE JSON line.  `value` = tokens/s of the whole job (inputs resident in
HBM), `e2e` = the same through the public API with the step's inputs copied
from pinned host memory and the losses read back, `roofline` for the dominant
kernel (CUDA events around each launch on its stream, inside the timed
region), `cpu_baseline` = the fp64 oracle on a bounded sample on the host.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Multi-GPU: one process per GPU (torchrun); every rank runs its own replica of
the step on its own micro-batches (weak scaling, no collective on the data
path); the step time is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused GRPO head fwd+bwd tokens/sec; TFLOPS as % of GB300 dense BF16 peak"
# Secondary workloads: name -> (workload index in synth.CONFIGS, storage dtype, what a step runs)
AUX_WORKLOADS = {
    "gspo_packed": (3, "bf16", "fwd+gspo+bwd"),
    "grpo_small": (2, "bf16", "fwd+grpo+bwd"),
    "selective_logp_bf16": (1, "bf16", "fwd"),
    "selective_logp_f32": (1, "fp32", "fwd"),
    "grpo_small_f32": (2, "fp32", "fwd+grpo+bwd"),
    "tiny_fp32_grpo": (0, "fp32", "fwd+grpo+bwd"),
}
# fp32 FMA peak of the SIMT twin: 152 SMs x 128 fp32 lanes x 2 FLOP x 2070 MHz
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.070e9 / 1e12
L2_FLUSH_BYTES = 512 << 20
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=8)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--micro-batches", type=int, default=None, help="override (testing only)")
    ap.add_argument("--cpu-rows", type=int, default=768,
                    help="tokens in the oracle's timed sample (about 12 s of host work on 16 Arm cores)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--graph", action="store_true",
                    help="secondary workloads: capture the step in a CUDA graph and time its replays")
    ap.add_argument("--workload", choices=["grpo_8b_vocab"] + sorted(AUX_WORKLOADS), default="grpo_8b_vocab",
                    help="grpo_8b_vocab (default) is the headline step; the others measure the remaining paths "
                         "(one GPU, L2 flushed between timed steps)")
    return ap.parse_args()


# ---------------------------------------------------------------- distributed
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def rank_micro_batches(rank: int, per_rank: int):
    """Micro-batch indices (seed streams) of one rank: disjoint across ranks."""
    return [rank * per_rank + k for k in range(per_rank)]


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        try:
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        finally:
            os.unlink(self.path)
        if not rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return float("nan")

        sm = [num(r[1]) for r in rows if not math.isnan(num(r[1]))]
        mx = max(num(r[2]) for r in rows)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(num(r[3]) for r in rows)}


def kernel_traffic(name: str):
    """DRAM bytes per launch of `name` from the committed ncu summary, or None
    when the kernel sources changed since that capture."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic_tc_kernels_8b_vocab.json")
    try:
        d = json.load(open(path))
        h = hashlib.sha256()
        for src in d["source_files"]:
            h.update(open(os.path.join(ROOT, src), "rb").read())
        if h.hexdigest() != d["source_sha256"]:
            return None
        k = d["kernels"][name]
        return int(k["dram_read_bytes"]) + int(k["dram_write_bytes"])
    except (OSError, KeyError, ValueError):
        return None


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]), float(d.get("hbm_gbs", 0)), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS, FALLBACK_BF16_TFLOPS_SUSTAINED, 6800.0, "fallback"


# ---------------------------------------------------------------- CPU oracle leg
_ORACLE_CACHE = {}


def o_n_bytes(name: str, N: int, splits: int, with_ref: bool):
    """Algorithmic HBM bytes of one launch of an O(N) kernel over N tokens: every
    input read once, every output written once (None for other kernels)."""
    if name == "merge_lse":        # part_m, part_s [splits, N]; zy, targets, mask -> logp, lse
        return 8 * splits * N + 17 * N
    if name == "grpo_loss":        # logp, old, ref, mask, seq_id -> coef
        return 21 * N
    if name == "gspo_segment":     # logp, old (, ref), mask, seg_id -> coef
        return (21 if with_ref else 17) * N
    return None


def add_o_n_rates(kernels: dict, N: int, splits: int, with_ref: bool, hbm: float):
    for name, ent in kernels.items():
        nb = o_n_bytes(name, N, splits, with_ref)
        if nb is None:
            continue
        sec = ent.get("avg_launch_ms", ent.get("avg_launch_us", 0) * 1e-3) * 1e-3
        ent["algorithmic_bytes"] = nb
        ent["gb_per_s"] = round(nb / sec / 1e9, 1) if sec > 0 else None
        ent["hbm_frac"] = round(nb / sec / 1e9 / hbm, 4) if sec > 0 and hbm > 0 else None


def oracle_sample(cfg, rows: int, norm: float):
    """Time the fp64 oracle on `rows` tokens of micro-batch 0 (full V and D):
    logits + LSE, GRPO loss terms and the dH / dW contributions of those rows.
    Input preparation (drawing and upcasting) is outside the timed part.
    Returns (tokens/s, seconds, cores, description)."""
    import oracle
    from synth import make_workload
    if "w" not in _ORACLE_CACHE:
        _ORACLE_CACHE["w"] = make_workload(cfg, N=cfg.N)
    w = _ORACLE_CACHE["w"]
    if "W" not in _ORACLE_CACHE:
        _ORACLE_CACHE["W"] = oracle.as_f64(w.pop("W"), "bf16")
    W = _ORACLE_CACHE["W"]
    H = oracle.as_f64(w["H"][:rows], "bf16")
    y, m, seq = w["targets"][:rows], w["mask"][:rows], w["seq_id"][:rows]
    adv = oracle.group_advantages(w["rewards"], w["group_size"])
    t0 = time.perf_counter()
    lp, lse, _ = oracle.selected_logprob(H, W, y, m)
    old = lp + w["u_old"][:rows]
    ref = lp + w["u_ref"][:rows]
    res = oracle.grpo_loss(lp, old, ref, m, seq, adv, w["num_seqs"], cfg.eps_low, cfg.eps_high, cfg.beta,
                           "token_mean", norm)
    dH, dW = oracle.head_backward(H, W, y, lse, res["coef"])
    dt = time.perf_counter() - t0
    del dH, dW
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    desc = (f"{rows} tokens of one 8192-token micro-batch, full V={cfg.V} and D={cfg.D}: fp64 logits + LSE, "
            f"GRPO loss, dH and dW contributions (numpy/OpenBLAS, all host cores)")
    return rows / dt, dt, cores, desc


# ---------------------------------------------------------------- GPU leg
def run_ours(args, rank, world, local):
    import numpy as np
    import torch

    import gspo_logprob_gb300 as g
    from gspo_logprob_gb300 import ops
    from synth import CONFIGS, make_workload

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init(world, "nccl")
    g.build()
    cfg = CONFIGS[4]
    MB = args.micro_batches or cfg.micro_batches
    N, D, V = cfg.N, cfg.D, cfg.V

    # ---- inputs (seeded, synthetic), resident in HBM
    mbs = rank_micro_batches(rank, MB)
    w0 = make_workload(cfg, micro_batch=mbs[0])
    W = torch.from_numpy(w0["W"].view(np.int16)).view(torch.bfloat16).to(dev)
    if rank == 0 and mbs[0] == 0:
        _ORACLE_CACHE["w"] = w0  # the CPU leg samples the same micro-batch (and W)
    host = []
    for k, mb in enumerate(mbs):
        w = w0 if k == 0 else make_workload(cfg, micro_batch=mb, with_weight=False)
        host.append(w)
    norm = float(sum(int(w["mask"].sum()) for w in host))  # the step's active tokens

    def t(x, bf=False):
        a = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16) if bf else \
            torch.from_numpy(np.ascontiguousarray(x))
        return a

    Hh = torch.stack([t(w["H"], True) for w in host]).pin_memory()
    yh = torch.stack([t(w["targets"]) for w in host]).pin_memory()
    mh = torch.stack([t(w["mask"]) for w in host]).pin_memory()
    sh = torch.stack([t(w["seq_id"]) for w in host]).pin_memory()
    rh = torch.stack([t(w["rewards"]) for w in host]).pin_memory()
    H, y, m, seq, rew = (x.to(dev) for x in (Hh, yh, mh, sh, rh))
    # old/ref log-probs: the configuration defines them as logp + U(-a, a); logp
    # comes from an untimed forward pass (as a previous policy pass would give it)
    old = torch.empty(MB, N, dtype=torch.float32, device=dev)
    ref = torch.empty(MB, N, dtype=torch.float32, device=dev)
    for k, w in enumerate(host):
        fw = g.grpo_head_forward(H[k], W, y[k], m[k])
        old[k] = fw["logp"] + torch.from_numpy(w["u_old"]).to(dev)
        ref[k] = fw["logp"] + torch.from_numpy(w["u_ref"]).to(dev)
    oldh, refh = old.cpu().pin_memory(), ref.cpu().pin_memory()
    nseq = host[0]["num_seqs"]
    G = host[0]["group_size"]

    dH = torch.empty(MB, N, D, dtype=torch.bfloat16, device=dev)
    dW = torch.empty(V, D, dtype=torch.float32, device=dev)
    loss3 = torch.empty(MB, 3, dtype=torch.float32, device=dev)
    clipped = torch.zeros(MB, dtype=torch.int32, device=dev)
    outs = [dict(logp=torch.empty(N, device=dev), lse=torch.empty(N, device=dev), coef=torch.empty(N, device=dev),
                 loss3=loss3[k], num_clipped=clipped[k:k + 1]) for k in range(MB)]
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    def micro_step(k, Hk, yk, mk, seqk, rewk, oldk, refk):
        adv = g.grpo_group_advantage(rewk, G, status=status)
        fw = g.grpo_head_forward(Hk, W, yk, mk, old_logp=oldk, ref_logp=refk, adv=adv, seq_id=seqk, num_seqs=nseq,
                                 eps_low=cfg.eps_low, eps_high=cfg.eps_high, beta=cfg.beta, norm=norm,
                                 clip_count=True, status=status, out=outs[k])
        g.grpo_head_backward(Hk, W, yk, mk, fw["lse"], fw["coef"], dH=dH[k], dW=dW, accumulate_dW=k > 0,
                             status=status)

    def step(Hs, ys, ms, seqs, rews, olds, refs):
        for k in range(MB):
            micro_step(k, Hs[k], ys[k], ms[k], seqs[k], rews[k], olds[k], refs[k])

    args_dev = (H, y, m, seq, rew, old, ref)
    for _ in range(args.warmup):
        step(*args_dev)
    torch.cuda.synchronize()
    ops.raise_on_status(status)
    torch.cuda.reset_peak_memory_stats(dev)
    base_mem = torch.cuda.memory_allocated(dev)

    # ---- timed region (device-resident inputs)
    clocks = ClockSampler(local)
    if rank == 0:
        clocks.start()
    ops.profile_reset()
    ops.profile_enable(True)
    n_launch0 = ops.launch_count()
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        step(*args_dev)
    e1.record()
    torch.cuda.synchronize()
    barrier(world)
    launches = ops.launch_count() - n_launch0
    ops.profile_enable(False)
    prof = ops.profile_read()
    clk = clocks.stop() if rank == 0 else None
    peak_mem = torch.cuda.max_memory_allocated(dev) - base_mem
    ops.raise_on_status(status)
    ms_step = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)

    # ---- end to end: pinned host inputs -> device, step, losses -> host.  A user
    # overlaps the upload of micro-batch k+1 (copy stream) with the compute of
    # micro-batch k (two input slots), and the next step's first upload with this
    # step's last micro-batch; every byte still crosses inside the timed region,
    # and each step ends with its losses read back on the host.
    e2e = None
    if not args.no_e2e:
        hosts = (Hh, yh, mh, sh, rh, oldh, refh)
        slots = [tuple(torch.empty(x.shape[1:], dtype=x.dtype, device=dev) for x in hosts) for _ in range(2)]
        copy_stream = torch.cuda.Stream(dev)
        comp = torch.cuda.current_stream(dev)
        copied = [torch.cuda.Event() for _ in range(2)]
        freed = [torch.cuda.Event() for _ in range(2)]
        for ev in freed:
            ev.record(comp)
        loss_h = torch.empty(MB, 3, dtype=torch.float32).pin_memory()
        h2d = sum(x.numel() * x.element_size() for x in hosts)
        d2h = loss_h.numel() * loss_h.element_size()

        def upload(k):
            s = k % 2
            with torch.cuda.stream(copy_stream):
                copy_stream.wait_event(freed[s])
                for b, hx in zip(slots[s], hosts):
                    b.copy_(hx[k], non_blocking=True)
                copied[s].record(copy_stream)

        def e2e_step(first_uploaded, prefetch_next):
            # micro-batch k uses slot k % 2 (MB is even, so the next step's
            # micro-batch 0 goes to slot 0 while this step's last one uses slot 1)
            if not first_uploaded:
                upload(0)
            for k in range(MB):
                if k + 1 < MB:
                    upload(k + 1)
                elif prefetch_next:
                    upload(0)
                comp.wait_event(copied[k % 2])
                micro_step(k, *slots[k % 2])
                freed[k % 2].record(comp)
            loss_h.copy_(loss3, non_blocking=True)
            torch.cuda.synchronize()

        total = args.warmup + args.steps
        prefetched = False
        for it in range(total):
            if it == args.warmup:
                barrier(world)
                torch.cuda.synchronize()
                t0 = time.perf_counter()
            # the timed region's first upload is its own; the last step prefetches nothing
            nxt = MB % 2 == 0 and it + 1 < total and it + 1 != args.warmup
            e2e_step(prefetched, nxt)
            prefetched = nxt
        wall = max_over_ranks((time.perf_counter() - t0) / args.steps, world, dev)
        ops.raise_on_status(status)
        e2e = {"value": world * MB * N / wall, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": wall * 1e3,
               "path": "gspo_logprob_gb300 binding -> C ABI; each micro-batch's inputs uploaded from pinned host "
                       "memory on a copy stream while the previous micro-batch computes; losses read back"}

    # ---- numbers
    tokens_step = world * MB * N
    flops_step = 8.0 * tokens_step * D * V
    burst, sustained, hbm, src = measured_peaks()
    tflops = flops_step / (ms_step * 1e-3) / 1e12
    alg = {  # algorithmic FLOPs per step of each kernel kind (real vocabulary columns)
        "fwd_logits_lse_tc": 2.0 * MB * N * D * V,
        "dlogits_tc": 2.0 * MB * N * D * V,
        "dh_gemm_tc": 2.0 * MB * N * D * V,
        "dw_gemm_tc": 2.0 * MB * N * D * V,
        "dhdw_gemm_tc": 4.0 * MB * N * D * V,   # dH and dW of a block in one launch
    }
    kernels = {}
    for name, (n, tot) in prof.items():
        per_step_ms = tot / args.steps
        ent = {"launches_per_step": n / args.steps, "ms_per_step": round(per_step_ms, 4),
               "avg_launch_ms": round(tot / n, 5), "share": round(per_step_ms / ms_step, 4)}
        if name in alg:
            ent["tflops"] = round(alg[name] / (per_step_ms * 1e-3) / 1e12, 1)
        kernels[name] = ent
    add_o_n_rates(kernels, N, -(-V // 256), True, hbm)
    dom = max((k for k in kernels if k in alg), key=lambda k: kernels[k]["ms_per_step"])
    dom_launches = kernels[dom]["launches_per_step"]
    roof = {"kernel": dom, "bound": "tensor", "achieved": kernels[dom]["tflops"], "peak": sustained,
            "unit": "TFLOP/s", "frac": round(kernels[dom]["tflops"] / sustained, 4), "traffic": kernel_traffic(dom),
            "traffic_unit": "bytes per launch (ncu dram read+write, one capture; null if the kernel changed)",
            "algorithmic_flops_per_launch": alg[dom] / dom_launches,
            "peak_source": f"{src} bf16_tflops_sustained (kernel timed inside a multi-second step)"}
    ws_bytes = max(ops.forward_workspace_bytes(ops.make_head(H[0], W, y[0], m[0])),
                   ops.backward_workspace_bytes(ops.make_head(H[0], W, y[0], m[0])))
    out = {
        "metric": METRIC, "value": round(tokens_step / (ms_step * 1e-3), 1), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "bf16 GRPO head at 8B-model scale: 16 prompts x G=8 x T=1024 = 131072 tokens/GPU in "
                               "16 micro-batches of 8192, D=4096, V=151936, token-mean (global normaliser), "
                               "eps 0.2/0.28, beta 0.04",
                   "tokens_per_step_per_gpu": MB * N, "micro_batch": N, "D": D, "V": V,
                   "l2": "inputs larger than L2 (W is 1.24 GB)", "parallelism": f"replicas x{world}"},
        "tflops": round(tflops, 1), "pct_of_peak": round(100 * tflops / burst, 2),
        "pct_of_sustained_peak": round(100 * tflops / sustained, 2),
        "peak_tflops": {"burst": burst, "sustained": sustained, "source": src},
        "roofline": roof,
        "kernels": kernels,
        "gpu_launches": launches,
        "peak_extra_mem": {"workspace_bytes": ws_bytes, "measured_peak_delta_bytes": int(peak_mem),
                           "NxVx2_bytes": N * V * 2, "workspace_frac": round(ws_bytes / (N * V * 2), 4),
                           "measured_frac": round(peak_mem / (N * V * 2), 4)},
        "clocks": clk,
        "e2e": e2e,
        "clip_fraction": {"clipped_tokens": int(clipped.sum().item()), "active_tokens": int(norm),
                          "value": round(int(clipped.sum().item()) / max(norm, 1.0), 6),
                          "what": "active tokens of the last step whose policy gradient the clip cuts off"},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tps, secs, cores, desc = oracle_sample(cfg, args.cpu_rows, norm)
        out["cpu_baseline"] = {"value": round(tps, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                               "sample": desc, "seconds": round(secs, 2)}
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------- secondary workloads
def oracle_sample_aux(cfg, w, dt: str, what: str, rows: int):
    """The fp64 oracle on `rows` tokens of workload `cfg` (the same inputs the
    GPU leg runs): logits + LSE, and for the loss workloads the loss over the
    whole batch plus the sampled rows' dH / dW contributions."""
    import numpy as np

    import oracle
    W = oracle.as_f64(w["W"], dt)
    H = oracle.as_f64(w["H"][:rows], dt)
    y, m, seq = w["targets"][:rows], w["mask"][:rows], w["seq_id"][:rows]
    t0 = time.perf_counter()
    lp, lse, _ = oracle.selected_logprob(H, W, y, m)
    if what != "fwd":
        adv = oracle.group_advantages(w["rewards"], w["group_size"])
        if cfg.kind == "gspo":
            lp_all = np.full(cfg.N, -math.log(cfg.V))
            lp_all[:rows] = lp
            res = oracle.gspo_loss(lp_all, lp_all + w["u_old"], w["mask"], w["seq_id"], cfg.num_docs, adv,
                                   cfg.eps_low, cfg.eps_high, float(cfg.num_docs))
            coef = res["coef"][:rows]
        else:
            res = oracle.grpo_loss(lp, lp + w["u_old"][:rows], lp + w["u_ref"][:rows], m, seq, adv, w["num_seqs"],
                                   cfg.eps_low, cfg.eps_high, cfg.beta, "token_mean")
            coef = res["coef"]
        oracle.head_backward(H, W, y, lse, coef)
    dt_s = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    desc = f"{rows} of {cfg.N} tokens, full V={cfg.V} and D={cfg.D}: fp64 {what.replace('+', ', ')} (numpy/OpenBLAS)"
    return rows / dt_s, dt_s, cores, desc


def run_aux(args, rank, world, local):
    """One GPU: the workload `args.workload` names, each timed step bracketed by
    CUDA events and followed (outside the events) by an L2 flush."""
    import numpy as np
    import torch

    import gspo_logprob_gb300 as g
    from gspo_logprob_gb300 import ops
    from synth import CONFIGS, make_workload

    if world > 1:
        raise SystemExit("secondary workloads run on one GPU")
    idx, dt, what = AUX_WORKLOADS[args.workload]
    cfg = CONFIGS[idx]
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    g.build()
    w = make_workload(cfg, dtype=dt)
    N, D, V = cfg.N, cfg.D, cfg.V

    def mat(x):
        a = torch.from_numpy(np.ascontiguousarray(x))
        return (a.view(torch.int16).view(torch.bfloat16) if dt == "bf16" else a).to(dev)

    H, W = mat(w["H"]), mat(w["W"])
    y, m = (torch.from_numpy(w[k]).to(dev) for k in ("targets", "mask"))
    seq = torch.from_numpy(w["seq_id"]).to(dev)
    status = ops.new_status(dev)
    out = dict(logp=torch.empty(N, device=dev), lse=torch.empty(N, device=dev))
    if what != "fwd":
        lp0 = g.grpo_head_forward(H, W, y, m)["logp"]
        old = lp0 + torch.from_numpy(w["u_old"]).to(dev).float()
        ref = lp0 + torch.from_numpy(w["u_ref"]).to(dev).float()
        rew = torch.from_numpy(w["rewards"]).to(dev)
        G, S = w["group_size"], w["num_seqs"]
        dH = torch.empty(N, D, dtype=H.dtype, device=dev)
        dW = torch.empty(V, D, dtype=torch.float32, device=dev)
        out.update(coef=torch.empty(N, device=dev), loss3=torch.empty(3, device=dev))

    last = {}  # the last step's clipped count (device tensor)
    head = ops.make_head(H, W, y, m)
    ws_f = torch.empty(ops.forward_workspace_bytes(head), dtype=torch.uint8, device=dev)
    ws_b = torch.empty(ops.backward_workspace_bytes(head), dtype=torch.uint8, device=dev)

    def step():
        if what == "fwd":
            g.grpo_head_forward(H, W, y, m, status=status, out=out, workspace=ws_f)
            return
        adv = g.grpo_group_advantage(rew, G, status=status)
        if cfg.kind == "gspo":
            fw = g.grpo_head_forward(H, W, y, m, status=status, out=out, workspace=ws_f)
            gs = g.gspo_segment_loss(fw["logp"], old, m, seq, S, adv, eps_low=cfg.eps_low, eps_high=cfg.eps_high,
                                     divisor=float(S), status=status)
            coef = gs["coef"]
            last["clipped"] = gs["num_clipped"]
        else:
            fw = g.grpo_head_forward(H, W, y, m, old_logp=old, ref_logp=ref, adv=adv, seq_id=seq, num_seqs=S,
                                     eps_low=cfg.eps_low, eps_high=cfg.eps_high, beta=cfg.beta, status=status,
                                     out=out, workspace=ws_f, clip_count=True)
            coef = fw["coef"]
            last["clipped"] = fw["num_clipped"]
        g.grpo_head_backward(H, W, y, m, fw["lse"], coef, dH=dH, dW=dW, status=status, workspace=ws_b)

    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        step()
        flush.zero_()
    torch.cuda.synchronize()
    ops.raise_on_status(status)
    per_replay = 0
    if args.graph:
        # one capture of the whole step; the timed loop replays it (no host work per kernel)
        graph = torch.cuda.CUDAGraph()
        n0 = ops.launch_count()
        with torch.cuda.graph(graph):
            step()
        per_replay = ops.launch_count() - n0
        eager_step = step

        def step():  # noqa: F811
            graph.replay()
        for _ in range(args.warmup):
            step()
            flush.zero_()
        torch.cuda.synchronize()
        ops.raise_on_status(status)
        del eager_step
    clocks = ClockSampler(local)
    clocks.start()
    ops.profile_reset()
    ops.profile_enable(True)
    n0 = ops.launch_count()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    torch.cuda.synchronize()
    for a, b in ev:
        a.record()
        step()
        b.record()
        flush.zero_()
    torch.cuda.synchronize()
    launches = ops.launch_count() - n0 + per_replay * args.steps
    ops.profile_enable(False)
    prof = ops.profile_read()
    clk = clocks.stop()
    ops.raise_on_status(status)
    ms_step = sum(a.elapsed_time(b) for a, b in ev) / args.steps

    passes = {"fwd": 1, "fwd+grpo+bwd": 4, "fwd+gspo+bwd": 4}[what]
    flops_step = 2.0 * passes * N * D * V
    burst, _, hbm, src = measured_peaks()
    if dt == "bf16":
        alg = {k: 2.0 * N * D * V for k in ("fwd_logits_lse_tc", "dlogits_tc", "dh_gemm_tc", "dw_gemm_tc")}
        alg["dhdw_gemm_tc"] = 4.0 * N * D * V
        bound, peak, peak_src = "tensor", burst, f"{src} bf16_tflops (burst: a short step timed alone)"
    else:
        alg = {"fwd_logits_lse_f32": 2.0 * N * D * V, "dlogits_f32": 2.0 * N * D * V, "gemm_f32": 4.0 * N * D * V}
        bound, peak = "alu", FP32_ALU_TFLOPS
        peak_src = "152 SMs x 128 fp32 lanes x 2 FLOP (FMA) x 2070 MHz maximum SM clock"
    kernels = {}
    for name, (n, tot) in prof.items():
        per_step_ms = tot / args.steps
        ent = {"launches_per_step": n / args.steps, "ms_per_step": round(per_step_ms, 5),
               "avg_launch_us": round(1e3 * tot / n, 2), "share": round(per_step_ms / ms_step, 4)}
        if name in alg:
            ent["tflops"] = round(alg[name] / (per_step_ms * 1e-3) / 1e12, 2)
        kernels[name] = ent
    add_o_n_rates(kernels, N, -(-V // 256), cfg.kind != "gspo", hbm)
    if kernels:
        dom = max((k for k in kernels if k in alg), key=lambda k: kernels[k]["ms_per_step"])
        roof = {"kernel": dom, "bound": bound, "achieved": kernels[dom]["tflops"], "peak": round(peak, 1),
                "unit": "TFLOP/s", "frac": round(kernels[dom]["tflops"] / peak, 4), "traffic": None,
                "algorithmic_flops_per_launch": alg[dom] / kernels[dom]["launches_per_step"], "peak_source": peak_src}
    else:
        # graph replays carry no per-launch events: the whole step against the roofline
        st_tf = flops_step / (ms_step * 1e-3) / 1e12
        roof = {"kernel": "whole step (CUDA graph replay)", "bound": bound, "achieved": round(st_tf, 2),
                "peak": round(peak, 1), "unit": "TFLOP/s", "frac": round(st_tf / peak, 4), "traffic": None,
                "algorithmic_flops_per_launch": flops_step, "peak_source": peak_src}
    res = {
        "metric": METRIC, "value": round(N / (ms_step * 1e-3), 1), "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if dt == "bf16" else "f32", "data": "synthetic",
        "config": {"workload": f"{args.workload}: shapes of {cfg.name}, N={N}, D={D}, V={V}, {dt}, step = {what}"
                               + (" (CUDA graph replay)" if args.graph else ""),
                   "l2": "flushed between timed steps (512 MB write outside the events)"},
        "tflops": round(flops_step / (ms_step * 1e-3) / 1e12, 2), "roofline": roof, "kernels": kernels,
        "gpu_launches": launches, "clocks": clk, "e2e": None,
        "peak_extra_mem": {"workspace_bytes": max(ws_f.numel(), ws_b.numel() if what != "fwd" else 0),
                           "NxVx2_bytes": N * V * 2,
                           "workspace_frac": round(max(ws_f.numel(), ws_b.numel() if what != "fwd" else 0)
                                                   / (N * V * 2), 4)},
    }
    if "clipped" in last:
        nclip = int(last["clipped"].item())
        if cfg.kind == "gspo":
            live = int(np.sum(np.bincount(w["seq_id"][(w["seq_id"] >= 0) & (w["mask"] > 0)],
                                          minlength=w["num_seqs"]) > 0))
            res["clip_fraction"] = {"clipped": nclip, "of": live, "value": round(nclip / max(live, 1), 4),
                                    "what": "live segments whose policy gradient the clip cuts off"}
        else:
            act = int(w["mask"].sum())
            res["clip_fraction"] = {"clipped": nclip, "of": act, "value": round(nclip / max(act, 1), 6),
                                    "what": "active tokens whose policy gradient the clip cuts off"}
    if not args.no_cpu_baseline:
        rows = {0: N, 1: N, 2: N, 3: 256}[idx]
        tps, secs, cores, desc = oracle_sample_aux(cfg, w, dt, what, rows)
        res["cpu_baseline"] = {"value": round(tps, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                               "sample": desc, "seconds": round(secs, 2)}
    print(json.dumps(res), flush=True)


def run_reference(args, rank, world):
    """The oracle as it stands, on the host cores, on bounded samples of the
    same workload (rank 0 only)."""
    if rank != 0:
        return
    from synth import CONFIGS, make_workload
    cfg = CONFIGS[4]
    host_masks = [make_workload(cfg, micro_batch=k, with_weight=False)["mask"] for k in range(cfg.micro_batches)]
    norm = float(sum(int(x.sum()) for x in host_masks))
    rows = max(8, args.cpu_rows // 4)
    for _ in range(max(0, min(args.warmup, 1))):
        oracle_sample(cfg, 8, norm)
    times = []
    for _ in range(args.steps):
        tps, secs, cores, desc = oracle_sample(cfg, rows, norm)
        times.append(secs)
    sec = sum(times) / len(times)
    v = rows / sec
    out = {"impl": "reference", "metric": METRIC, "value": round(v, 3), "unit": "tokens/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 1), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": "bf16 GRPO head at 8B-model scale (same inputs), each step a bounded sample of "
                                  f"{rows} tokens", "D": cfg.D, "V": cfg.V, "parallelism": "host cores"},
           "cpu_baseline": {"value": round(v, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                            "sample": desc},
           "e2e": {"value": round(v, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.workload != "grpo_8b_vocab":
        run_aux(args, rank, world, local)
        return
    run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
