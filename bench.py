#!/usr/bin/env python
"""Benchmark of the DFlash drafter hot path on GB300.

One step = one draft+accept step over the batch, all of it on the GPU:
  draft_block (embed, n_l draft layers, final norm, LM head + argmax)
  -> planted target ids (synthetic stand-in for the target's verify forward)
  -> verify_accept (longest matching prefix, state advance by the accepted count).
Metric: draft blocks/s (= batch / step time) with microseconds per step and
the fraction of the 8 TB/s HBM roofline (weight + context KV bytes / time).
The context append of the n+1 committed rows (fc + RMSNorm + every layer's
K/V) runs between timed steps, and the whole iteration (draft + verify +
append) is timed as well.  Steps replay captured CUDA graphs; the weights
(1.8 GB) are larger than L2, so no L2 flush is needed.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config NAME] [--K K]
Multi-GPU (torchrun): each rank runs its own batch (independent sequences, no
collective on the data path), value = blocks/s summed over ranks (weak scaling).
"""
from __future__ import annotations

import argparse
import json
import os
import platform
import subprocess
import tempfile
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "draft blocks/s & µs per draft+accept step at K=16; % of 8 TB/s HBM roofline"
NOMINAL_HBM_GBS = 8000.0


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# sources of the LM-head kernels (the partial-store GEMM and the argmax kernel)
KERNEL_SOURCES = ("gemm_tc.cu", "elementwise.cu", "epilogue.cuh", "common.cuh", "internal.h")


def kernel_hash():
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "block_diffusion_speculative_dflash_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def lm_traffic(s, K):
    """DRAM bytes of one LM-head launch from the committed ncu summary, if it was
    taken on this workload with the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "lmhead_gemm_tc_argmax_qwen3_4b.md")
    try:
        kv = {}
        with open(path) as f:
            for line in f:
                if line.startswith("<!-- ") and ":" in line:
                    k, v = line[5:].split("-->")[0].split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("sources") != kernel_hash() or kv.get("workload") != f"{s.name} K={K}":
            return None
        return float(kv["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


def other_config_cmd(name, steps=8, warmup=3):
    """The bench command of another workload, run in a child process beside the headline
    (the same script and path, its own CUDA context; no CPU baseline, e2e or K sweep)."""
    return [sys.executable, os.path.abspath(__file__), "--config", name, "--steps", str(steps),
            "--warmup", str(warmup), "--no-cpu-baseline", "--no-e2e", "--k-sweep=", "--other-configs="]


def other_config_summary(name, rc, stdout, stderr=""):
    """What the headline line reports of another workload's run: its step time, blocks/s,
    clocks and workload from the last JSON line the child printed, or why there is none."""
    line = None
    for text in reversed((stdout or "").splitlines()):
        text = text.strip()
        if text.startswith("{"):
            try:
                line = json.loads(text)
                break
            except ValueError:
                continue
    if rc != 0 or line is None or "ms_per_step" not in line:
        tail = " | ".join(((stderr or "") + "\n" + (stdout or "")).strip().splitlines()[-3:])
        return {"error": f"exit {rc}: {tail}"[:300]}
    return {"us_per_step": line["ms_per_step"] * 1e3, "blocks_per_s": line["value"],
            "clocks": line.get("clocks"), "workload": line.get("config", {}).get("workload"),
            "command": " ".join(["python bench.py"] + other_config_cmd(name)[2:])}


def run_other_configs(names, timeout=300):
    out = {}
    for name in names:
        try:
            r = subprocess.run(other_config_cmd(name), capture_output=True, text=True, timeout=timeout, cwd=ROOT)
            out[name] = other_config_summary(name, r.returncode, r.stdout, r.stderr)
        except Exception as e:   # (a timeout or a failed start: reported, not fatal to the headline)
            out[name] = {"error": f"{type(e).__name__}: {e}"[:300]}
    return out


def aggregate_ranks(ms_da, ms_it, B, world, device="cpu"):
    """Whole-job figures over `world` ranks that each ran their own batch of B
    independent sequences: the step time is the slowest rank's (max over ranks),
    and the job drafts B * world blocks in that time (weak scaling).  Only the
    two timings cross ranks; no data-path collective."""
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([ms_da, ms_it], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_da, ms_it = float(t[0].item()), float(t[1].item())
    return ms_da, ms_it, B * world / (ms_da / 1e3)


def step_bytes(s, ctx_lens, K, conditioning="kv"):
    """Algorithmic bytes of one iteration: every weight read once + context KV read + appended KV rows.

    Draft: n_l layer weights + LM head + KV of (c_b + R) slots per layer (K and V;
    R slots only without context K/V injection).
    Append: W_fc + every layer's [W_k; W_v] (feature rows and KV writes are < 0.1%);
    W_fc only with input fusion, nothing without context."""
    esz = 2 if s.dtype == "bf16" else 4
    H, I = s.hidden, s.intermediate
    layer = (s.q_dim + 2 * s.kv_dim) * H + H * s.q_dim + 2 * I * H + H * I
    draft_w = (s.n_layers * layer + s.vocab * H) * esz
    ctx_keys = (lambda c: int(c)) if conditioning == "kv" else (lambda c: 0)
    kv = sum(ctx_keys(c) + K + 1 for c in ctx_lens) * s.n_layers * 2 * s.kv_dim * esz
    append_w = {"kv": (H * s.feat_dim + s.n_layers * 2 * s.kv_dim * H) * esz,
                "input": H * s.feat_dim * esz, "none": 0}[conditioning]
    return draft_w + kv, append_w


class Clocks:
    """nvidia-smi sampler running during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, uuid: str):
        self.index = index
        self.uuid = uuid
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"dflash_clocks_{os.getpid()}_rank{index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.uuid}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def dev(a):
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def feats_rows(s, rows, rows_max, tag):
    from synth import make_features
    B = len(rows)
    out = np.zeros((B, rows_max, s.feat_dim), np.uint16 if s.dtype == "bf16" else np.float32)
    for b in range(B):
        if rows[b]:
            out[b, :rows[b]] = make_features(s, int(rows[b]), tag=tag, batch_index=b)
    return out


# --------------------------------------------------------------------------- CPU oracle

def cpu_oracle_run(s, K, steps, warmup, seq_limit=None, conditioning="kv"):
    """Time the oracle (fp32, numpy BLAS on every host core) on full iterations.

    Returns (seconds per step, sample description, cores)."""
    import oracle as orc
    from synth import (context_lengths, draw_accept_lengths, make_target_fill, make_weights, plant_targets)
    cores = len(os.sched_getaffinity(0))
    B = s.batch if seq_limit is None else min(seq_limit, s.batch)
    W = make_weights(s)
    ctx = context_lengths(s)[:B]
    dr = orc.OracleDrafter(s, W, B, dtype=np.float32, conditioning=conditioning)
    f = feats_rows(s, ctx, int(ctx.max()), "prefill")
    for b in range(B):
        dr.ctx_append(b, f[b, :ctx[b]])
    for b in range(B):
        dr.set_anchor(b, 1 + b)
    T = steps + warmup
    L = draw_accept_lengths(s, T, K)
    fill = make_target_fill(s, T, K)
    times = []
    for t in range(T):
        t0 = time.perf_counter()
        d, _ = dr.draft(K, want_logits=False)
        g = plant_targets(d, L[t, :B], fill[t, :B], s.vocab)
        n, _ = dr.verify(d, g)
        fs = feats_rows(s, n + 1, K + 1, f"step{t}")
        for b in range(B):
            dr.ctx_append(b, fs[b, :n[b] + 1])
        if t >= warmup:
            times.append(time.perf_counter() - t0)
    sample = (f"{B} of {s.batch} sequence(s) of the workload, {steps} full iterations "
              f"(draft + verify + append) after {warmup} warm-up, oracle in fp32; the GPU `value` times "
              f"draft + verify without the append, its `iteration` figure includes it")
    return float(np.mean(times)), sample, cores, B


# --------------------------------------------------------------------------- main

def target_verify_bench(args):
    """Target-side verify forward vs block width R = K + 1 (the pages' "K-flat"
    observation): a Llama-3.1-8B-shaped bf16 target (32 layers, H 4096, 32q/8kv
    x 128, I 14336, V 128256, theta 5e5), random N(0, 0.02) weights drawn on the
    device (seeded), batch 1 after a 2048-token prefill; each R's forward is
    captured once and replayed between CUDA events, never committed, so every
    replay sees the same cache.  Prints one JSON line."""
    import torch
    from block_diffusion_speculative_dflash_gb300 import DFlashTarget, TargetConfig
    from synth.configs import DrafterShape
    torch.cuda.set_device(0)
    s = DrafterShape(name="llama31_8b_target", hidden=4096, n_target_layers=5, n_layers=32, n_q_heads=32,
                     n_kv_heads=8, head_dim=128, intermediate=14336, vocab=128256, rope_theta=5e5, dtype="bf16",
                     batch=1, K=16, K_max=1024, seed=6)
    Rs = [int(r) for r in args.target_r.split(",")]
    r_max, ctx = max(max(Rs), 1024), 2048
    gen = torch.Generator(device="cuda")
    gen.manual_seed(6000)
    from synth.inputs import weight_shapes
    Wd = {}
    for name, shp in weight_shapes(s).items():
        if name in ("w_fc", "fc_norm"):
            continue
        if len(shp) == 1:   # norm gains 1
            Wd[name] = torch.ones(shp, dtype=torch.bfloat16, device="cuda")
        else:
            Wd[name] = (torch.randn(shp, generator=gen, device="cuda") * 0.02).to(torch.bfloat16)
    wbytes = sum(t.numel() * 2 for n, t in Wd.items() if n != "embed")   # the forward reads every matrix but E
    feat = [1, 8, 15, 22, 29]   # five layers from shallow to deep: the drafter's L_t = 5 features
    tg = DFlashTarget(TargetConfig.from_shape(s, r_max, feat_layers=feat), Wd, 1)
    stream = torch.cuda.current_stream()
    for c0 in range(0, ctx, r_max):   # prefill, kept
        n = min(r_max, ctx - c0)
        toks = torch.randint(0, s.vocab, (1, n), generator=gen, device="cuda", dtype=torch.int32)
        ids = torch.empty((1, n), dtype=torch.int32, device="cuda")
        tg.forward(toks, ids)
        tg.commit(np.array([n], np.int32))
    torch.cuda.synchronize()
    peak, peak_kind = peaks()
    rows = []
    for R in Rs:
        toks = torch.randint(0, s.vocab, (1, R), generator=gen, device="cuda", dtype=torch.int32)
        ids = torch.empty((1, R), dtype=torch.int32, device="cuda")
        feats = torch.empty((1, R, len(feat) * s.hidden), dtype=torch.bfloat16, device="cuda")
        tg.forward(toks, ids, feats=feats)   # sizes every workspace
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            tg.forward(toks, ids, feats=feats)
        for _ in range(args.warmup):
            g.replay()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for ea, eb in evs:
            ea.record(stream)
            g.replay()
            eb.record(stream)
        torch.cuda.synchronize()
        ms = float(np.median([ea.elapsed_time(eb) for ea, eb in evs]))
        kv = 32 * 2 * 8 * 128 * 2 * (ctx + R)   # the cache read by attention, every layer
        rows.append({"R": R, "K": R - 1, "us": ms * 1e3, "weights_gbs": wbytes / (ms / 1e3) / 1e9,
                     "frac_of_measured": (wbytes + kv) / (ms / 1e3) / 1e9 / peak})
        del g
    tg.query()   # raises on any device fault bit
    r16 = next((r for r in rows if r["R"] == 17), rows[0])
    line = {"metric": "target verify forward us per block vs R = K + 1 (K-flat); Llama-3.1-8B shape",
            "value": r16["us"], "unit": "us", "higher_is_better": False, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "llama31_8b target: 32 layers H=4096 32q/8kv x128 I=14336 V=128256 bf16, "
                                   "batch 1, context 2048, features of layers 1/8/15/22/29",
                       "weights_gb": wbytes / 1e9, "peak_gbs": peak, "peak_source": peak_kind},
            "per_R": rows,
            "flatness": {f"R{r['R']}/R{rows[0]['R']}": r["us"] / rows[0]["us"] for r in rows}}
    print(json.dumps(line), flush=True)


def k_sweep_bench(Wd, K_list, steps: int, warmup: int):
    """Draft + accept step time against the block length at context 4096 (the
    K-sweep workload), with the weights already on the device (the Qwen3-4B
    shape; their values do not change a timing).  One drafter, a captured
    draft + accept graph per K replayed between CUDA events, the context append
    of the committed rows replayed between the timed spans."""
    import torch
    from block_diffusion_speculative_dflash_gb300 import DFlashDrafter, DrafterConfig, plant_targets
    from synth import CONFIGS, context_lengths, draw_accept_lengths, make_target_fill
    s = CONFIGS["qwen3_4b_ksweep"].with_(K_max=max(K_list))
    B, Rm = s.batch, max(K_list) + 1
    ctx = context_lengths(s)
    T = len(K_list) * (steps + warmup + 2) + 4
    pool = int(sum(1 << int(np.ceil(np.log2(max(64, int(c) + (T + 4) * Rm + Rm)))) for c in ctx)) * 2
    dr = DFlashDrafter(DrafterConfig.from_shape(s, kv_pool_tokens=pool), Wd, B)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(2000 + s.seed)
    f0 = torch.randn((B, int(ctx.max()), s.feat_dim), generator=gen, device="cuda").to(torch.bfloat16)
    dr.ctx_append(f0, int(ctx.max()), rows=ctx.astype(np.int32))
    del f0
    dr.reserve_headroom((T + 4) * Rm + Rm)
    stream = torch.cuda.current_stream()
    out = {}
    first = True
    for K in K_list:
        R = K + 1
        L_tab = dev(draw_accept_lengths(s.with_(K=K), steps + warmup + 2, K))
        fill_tab = dev(make_target_fill(s.with_(K=K), steps + warmup + 2, K))
        ctr = torch.zeros(1, dtype=torch.int32, device="cuda")
        fstep = dev(feats_rows(s, [R] * B, R, "step"))
        d_ids = torch.zeros((B, K), dtype=torch.int32, device="cuda")
        g_ids = torch.zeros((B, R), dtype=torch.int32, device="cuda")
        acc = torch.zeros(B, dtype=torch.int32, device="cuda")
        nxt = torch.zeros(B, dtype=torch.int32, device="cuda")
        rows = torch.zeros(B, dtype=torch.int32, device="cuda")

        def draft_accept():
            dr.draft_block(K, draft_ids=d_ids)
            plant_targets(d_ids, L_tab, fill_tab, B, K, s.vocab, g_ids, step_counter=ctr, n_plans=steps + warmup + 2)
            dr.verify_accept(g_ids, accept_len=acc, next_anchor=nxt)

        def append():
            torch.add(acc, 1, out=rows)
            dr.ctx_append(fstep, R, rows=rows)

        dr.draft_block(K, anchor_ids=dev(np.arange(1, B + 1, dtype=np.int32)) if first else None, draft_ids=d_ids)
        first = False
        plant_targets(d_ids, L_tab, fill_tab, B, K, s.vocab, g_ids, step_counter=ctr, n_plans=steps + warmup + 2)
        dr.verify_accept(g_ids, accept_len=acc, next_anchor=nxt)
        append()
        torch.cuda.synchronize()
        g_da, g_ap = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_da):
            draft_accept()
        with torch.cuda.graph(g_ap):
            append()
        for _ in range(warmup):
            g_da.replay()
            g_ap.replay()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for ea, eb in evs:
            ea.record(stream)
            g_da.replay()
            eb.record(stream)
            g_ap.replay()
        torch.cuda.synchronize()
        out[str(K)] = round(float(np.mean([ea.elapsed_time(eb) for ea, eb in evs])) * 1e3, 1)
        del g_da, g_ap
    dr.query_state()
    dr.close()
    return {"us_per_step": out, "context": int(ctx.max()), "steps": steps, "warmup": warmup,
            "k128_over_k16": round(out["128"] / out["16"], 3) if "128" in out and "16" in out else None,
            "what": "draft + accept step of the Qwen3-4B-shaped drafter at context 4096, per K (mask tokens)"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="qwen3_4b")
    ap.add_argument("--K", type=int, default=None)
    ap.add_argument("--cpu-steps", type=int, default=3)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--target-verify", action="store_true",
                    help="time the target-side verify forward against the block width instead")
    ap.add_argument("--target-r", default="1,2,9,17,33,65,129,257,513,1025")
    ap.add_argument("--k-sweep", default="16,32,64,128",
                    help="block lengths of the context-4096 K sweep reported beside the headline ('' to skip)")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch (a smaller case, e.g. for a profiler capture)")
    ap.add_argument("--ctx-max", type=int, default=None,
                    help="cap the workload's context lengths (a smaller case, e.g. for a profiler capture)")
    ap.add_argument("--other-configs", default="llama31_8b,qwen3_4b_serving",
                    help="workloads also timed, each in a child process, and reported under "
                         "'other_configs' of the headline line ('' to skip)")
    ap.add_argument("--conditioning", default="kv", choices=["kv", "input", "none"],
                    help="how the target context conditions the draft: K/V injection (the method), "
                         "input fusion or none (the ablation variants)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.target_verify:
        return target_verify_bench(args)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    from synth import CONFIGS
    s = CONFIGS[args.config]
    if args.batch:
        s = s.with_(batch=args.batch)
    if args.ctx_max:
        kind, *lim = s.ctx
        s = s.with_(ctx=(kind, *[min(int(v), args.ctx_max) for v in lim]))
    K = args.K or s.K
    if K > s.K_max:
        s = s.with_(K_max=K)
    workload = (f"{args.config}: {s.n_layers}-layer drafter H={s.hidden} {s.n_q_heads}q/{s.n_kv_heads}kv x"
                f"{s.head_dim} I={s.intermediate} V={s.vocab} L_t={s.n_target_layers} {s.dtype}, batch {s.batch}, "
                f"context {s.ctx}, K={K}; step = draft + verify (planted targets)"
                + ("" if args.conditioning == "kv" else f"; conditioning: {args.conditioning}"))

    if args.impl == "reference":
        if rank != 0:
            return
        sec, sample, cores, Bs = cpu_oracle_run(s, K, args.steps, args.warmup, conditioning=args.conditioning)
        v = Bs / sec
        line = {"metric": METRIC, "value": v, "unit": "blocks/s", "n_gpus": args.gpus, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f32", "data": "synthetic",
                "config": {"workload": workload, "impl": "CPU oracle (numpy fp32)"},
                "impl": "reference",
                "cpu_baseline": {"value": v, "unit": "blocks/s", "cores": cores, "kind": "oracle", "sample": sample},
                "e2e": {"value": v, "unit": "blocks/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    import torch
    torch.cuda.set_device(local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    from block_diffusion_speculative_dflash_gb300 import DFlashDrafter, DrafterConfig, plant_targets
    from block_diffusion_speculative_dflash_gb300.binding import TRACE_APPEND, TRACE_DRAFT, TRACE_GEMM, TRACE_VERIFY
    from synth import context_lengths, draw_accept_lengths, make_target_fill, make_weights

    B, R = s.batch, K + 1
    W = make_weights(s)
    Wd = {k: dev(v) for k, v in W.items()}
    del W
    ctx = context_lengths(s)
    T = args.warmup + args.steps + 8
    cap = int(ctx.max()) + (T + 4) * R + R
    pool = int(sum(1 << int(np.ceil(np.log2(max(64, int(c) + (T + 4) * R + R)))) for c in ctx)) * 2
    dr = DFlashDrafter(DrafterConfig.from_shape(s, kv_pool_tokens=pool, conditioning=args.conditioning), Wd, B)
    stream = torch.cuda.current_stream()

    # prefill with seeded features generated on the device (padded host features
    # of the serving batch would be 26 GB), in one append when they fit in 32 GB
    # of device memory (one capacity allocation per sequence), else in chunks
    gen = torch.Generator(device="cuda")
    gen.manual_seed(1000 + s.seed)
    tdt = torch.bfloat16 if s.dtype == "bf16" else torch.float32
    esz = 2 if s.dtype == "bf16" else 4
    chunk = int(ctx.max()) if B * int(ctx.max()) * s.feat_dim * esz <= (32 << 30) else 4096
    for c0 in range(0, int(ctx.max()), chunk):
        rows_c = np.clip(ctx - c0, 0, chunk).astype(np.int32)
        n = int(rows_c.max())
        f0 = torch.randn((B, n, s.feat_dim), generator=gen, device="cuda").to(tdt)
        dr.ctx_append(f0, n, rows=rows_c)
        del f0
    dr.reserve_headroom((T + 4) * R + R)
    anchors = dev(np.arange(1, B + 1, dtype=np.int32))

    # per-step device inputs
    L_tab = dev(draw_accept_lengths(s, T, K))
    fill_tab = dev(make_target_fill(s, T, K))
    step_ctr = torch.zeros(1, dtype=torch.int32, device="cuda")
    fstep = dev(feats_rows(s, [R] * B, R, "step"))
    d_ids = torch.zeros((B, K), dtype=torch.int32, device="cuda")
    g_ids = torch.zeros((B, R), dtype=torch.int32, device="cuda")
    acc = torch.zeros(B, dtype=torch.int32, device="cuda")
    nxt = torch.zeros(B, dtype=torch.int32, device="cuda")
    rows = torch.zeros(B, dtype=torch.int32, device="cuda")

    def draft_accept():
        dr.draft_block(K, draft_ids=d_ids)
        plant_targets(d_ids, L_tab, fill_tab, B, K, s.vocab, g_ids, step_counter=step_ctr, n_plans=T)
        dr.verify_accept(g_ids, accept_len=acc, next_anchor=nxt)

    def append():
        torch.add(acc, 1, out=rows)
        dr.ctx_append(fstep, R, rows=rows)

    def step():
        draft_accept()
        append()

    # eager warm-up step (sets anchors, sizes every workspace), then capture
    dr.draft_block(K, anchor_ids=anchors, draft_ids=d_ids)
    plant_targets(d_ids, L_tab, fill_tab, B, K, s.vocab, g_ids, step_counter=step_ctr, n_plans=T)
    dr.verify_accept(g_ids, accept_len=acc, next_anchor=nxt)
    append()
    torch.cuda.synchronize()
    l0 = dr.launch_count()
    step()
    torch.cuda.synchronize()
    launches_per_step = dr.launch_count() - l0 + 1     # + the planting harness kernel
    # Timed graphs carry no trace events (an event node between two kernels turns
    # their programmatic overlap into a full dependency).  The headline replays
    # the draft+accept graph between two events, the append graph after it; the
    # iteration figure replays one graph of the whole step; an identical graph
    # with an event pair around every GEMM and API call gives per-kernel times.
    g_da, g_ap, g_full = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_da):
        draft_accept()
    with torch.cuda.graph(g_ap):
        append()
    with torch.cuda.graph(g_full):
        step()
    dr.trace_enable(4096)
    graph_tr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_tr):
        step()
    for _ in range(args.warmup):
        g_da.replay()
        g_ap.replay()
    g_full.replay()
    graph_tr.replay()
    torch.cuda.synchronize()
    dr.query_state()                                    # raises if any device fault bit is set
    st0 = dr.query_state()

    uuid = str(torch.cuda.get_device_properties(local_rank).uuid)
    clocks = Clocks(local_rank, uuid if uuid.startswith("GPU-") else f"GPU-{uuid}")
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for ea, eb in evs:
        ea.record(stream)
        g_da.replay()
        eb.record(stream)
        g_ap.replay()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        g_full.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    da = np.array([ea.elapsed_time(eb) for ea, eb in evs])
    ms_da = float(da.mean())
    ms_it = e0.elapsed_time(e1) / args.steps
    st1 = dr.query_state()
    # per-kernel durations: the traced graph, read after its last replay
    tr_steps = min(args.steps, 20)
    t0e = torch.cuda.Event(enable_timing=True)
    t1e = torch.cuda.Event(enable_timing=True)
    t0e.record(stream)
    for _ in range(tr_steps):
        graph_tr.replay()
    t1e.record(stream)
    torch.cuda.synchronize()
    ms_traced_step = t0e.elapsed_time(t1e) / tr_steps
    kinds, tms, tbytes = dr.trace_read()                # events of the last traced replay
    ms_da, ms_it, value = aggregate_ranks(ms_da, ms_it, B, world, device="cuda")

    # bytes: mean context over the timed steps (two passes of `steps` iterations)
    ctx_mid = (st0["ctx_len"] + st1["ctx_len"]) / 2.0
    draft_bytes, append_bytes = step_bytes(s, ctx_mid, K, args.conditioning)
    gem = kinds == TRACE_GEMM
    peak, peak_kind = peaks()
    # dominant kernel: the LM head (the largest single weight stream of the step)
    i_lm = int(np.argmax(np.where(gem, tbytes, -1.0)))
    lm_ms, lm_bytes = float(tms[i_lm]), float(tbytes[i_lm])
    achieved = lm_bytes / (lm_ms / 1e3) / 1e9 if lm_ms > 0 else None
    traffic = lm_traffic(s, K)
    da_gbs = draft_bytes / (ms_da / 1e3) / 1e9
    it_gbs = (draft_bytes + append_bytes) / (ms_it / 1e3) / 1e9
    lm_kernel = ("gemm_tc_kernel (LM head: tcgen05 weight stream, fp32 partial store; the argmax kernel after it "
                 "is not in this figure)" if s.dtype == "bf16" else "gemm_simt_kernel (LM head)")

    out = {
        "metric": METRIC, "value": value, "unit": "blocks/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_da, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": s.dtype, "data": "synthetic",
        "config": {"workload": workload, "global_batch": B * world, "K": K, "l2": "inputs larger than L2 (no flush)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "timing": "step = draft_block + verify_accept (planted targets); CUDA events around each "
                             "replay of its captured graph, the context append replayed between timed spans"},
        "us_per_step": ms_da * 1e3,
        "us_per_step_p90": float(np.percentile(da, 90)) * 1e3,
        "draft_accept_hbm_gbs": da_gbs,
        "draft_accept_frac_of_8tbs": da_gbs / NOMINAL_HBM_GBS,
        "draft_accept_frac_of_measured": da_gbs / peak,
        "bytes_per_step": draft_bytes,
        "iteration": {"us": ms_it * 1e3, "blocks_per_s": B * world / (ms_it / 1e3), "hbm_gbs": it_gbs,
                      "frac_of_8tbs": it_gbs / NOMINAL_HBM_GBS,
                      "what": "draft + verify + ctx_append of the n+1 committed rows, one captured graph"},
        "roofline": {"kernel": lm_kernel, "bound": "hbm", "achieved": achieved, "peak": peak,
                     "peak_source": "measured copy bandwidth (MEASURED_PEAKS.json hbm_gbs; burst)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "unit": "GB/s", "frac": achieved / peak if achieved else None,
                     "traffic": traffic,
                     "bytes_per_launch": lm_bytes, "launch_us": lm_ms * 1e3,
                     "timing": "CUDA event pair around the launch on its stream, traced replay of the step"},
        "gemms": {"launches_per_step": int(gem.sum()),
                  "each_us": [round(float(x) * 1e3, 2) for x in tms[gem]],
                  "each_gbs": [round(float(b) / float(t) / 1e6) for b, t in zip(tbytes[gem], tms[gem])]},
        "traced_us_per_iteration": ms_traced_step * 1e3,
        "gpu_launches": int(launches_per_step * args.steps),
        "launches_per_step": int(launches_per_step),
        "clocks": clk,
        "accept_mean": float(np.mean((st1["ctx_len"] - st0["ctx_len"]) / (2 * args.steps) - 1)),
    }

    # ---- end to end through the C-ABI with host buffers ----------------------------
    # The same step as `value` (draft, the device-side target harness, verify)
    # plus what a user's loop moves across the bus: the feature rows of the
    # accepted tokens in from pinned host memory (the append that the next draft
    # needs) and each step's accept lengths and next anchors out, read by the host
    # after one synchronisation per step.
    if not args.no_e2e:
        dr2 = dr
        dr2.trace_enable(0)   # the per-kernel event pairs above are instrumentation, not the user's loop
        pin = lambda a: torch.from_numpy(a).pin_memory()  # noqa: E731
        f_host = pin(feats_rows(s, [R] * B, R, "step").view(np.int16) if s.dtype == "bf16"
                     else feats_rows(s, [R] * B, R, "step"))
        acc_h = torch.zeros(B, dtype=torch.int32).pin_memory()
        nxt_h = torch.zeros(B, dtype=torch.int32).pin_memory()
        rows_h = torch.zeros(B, dtype=torch.int32).pin_memory()
        n_pl = args.e2e_steps + 3
        L2 = dev(draw_accept_lengths(s, n_pl, K, stream=1))
        fill2 = dev(make_target_fill(s, n_pl, K, stream=1))
        ctr2 = torch.zeros(1, dtype=torch.int32, device="cuda")
        dr2.reserve_headroom((args.e2e_steps + 4) * R + R)

        def e2e_step():
            dr2.draft_block(K, draft_ids=d_ids)
            plant_targets(d_ids, L2, fill2, B, K, s.vocab, g_ids, step_counter=ctr2, n_plans=n_pl)
            dr2.verify_accept(g_ids, accept_len=acc_h, next_anchor=nxt_h)
            stream.synchronize()
            rows_h.numpy()[:] = acc_h.numpy() + 1
            dr2.ctx_append(f_host, R, rows=rows_h)

        for _ in range(3):
            e2e_step()
        stream.synchronize()
        t0 = time.perf_counter()
        for _ in range(args.e2e_steps):
            e2e_step()
        stream.synchronize()
        sec = (time.perf_counter() - t0) / args.e2e_steps
        h2d = B * R * s.feat_dim * (2 if s.dtype == "bf16" else 4) + B * 4
        d2h = 2 * B * 4
        out["e2e"] = {"value": B * world / sec, "unit": "blocks/s", "h2d_bytes_per_step": h2d,
                      "d2h_bytes_per_step": d2h, "ms_per_step": sec * 1e3,
                      "note": "through the C-ABI: draft -> device target harness -> verify -> accept lengths and "
                              "next anchors to pinned host memory (one synchronisation) -> append of the "
                              "accepted rows' features from pinned host memory; copies and the sync timed"}
        dr2.query_state()

    # ---- the K sweep at context 4096 (the flatness of the step against K) -----------
    if args.k_sweep and args.config == "qwen3_4b" and args.conditioning == "kv" and world == 1:
        dr.close()
        torch.cuda.synchronize()
        out["k_sweep"] = k_sweep_bench(Wd, [int(k) for k in args.k_sweep.split(",")], steps=min(args.steps, 10),
                                       warmup=3)

    # ---- the other workloads' steps, each in a child process (rank 0, N=1 only) --------
    if args.other_configs and args.config == "qwen3_4b" and args.conditioning == "kv" and world == 1:
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        out["other_configs"] = run_other_configs([n for n in args.other_configs.split(",") if n])

    # ---- CPU oracle baseline on a bounded sample (rank 0, N=1 only) -----------------
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        sec, sample, cores, Bs = cpu_oracle_run(s, K, args.cpu_steps, 1, seq_limit=1, conditioning=args.conditioning)
        out["cpu_baseline"] = {"value": Bs / sec, "unit": "blocks/s", "cores": cores, "kind": "oracle",
                               "sample": sample, "cpu": platform.processor() or platform.machine()}
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
