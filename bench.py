"""Benchmark of the block-drafter hot path: draft tokens/s of (draft block + constrained argmax + verify).

Default workload: text speculative mode at the 4B-target drafter shape, batch 1, context 2048, block 16
(1 anchor + 15 proposals), vocabulary 151936, unconstrained, greedy verification against a synthetic target
row whose agreement prefix is Geometric(0.25).  The context K/V is prepared once before timing (its time is
reported separately).  All inputs are seeded synthetic data; the drafter weights (1.83 GB streamed per
block) are far larger than the 129 MB L2, so every step reads them from HBM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

N > 1 runs N independent replicas (one per rank, launched by torchrun): the path has no exchange step.
Prints ONE JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "draft tokens/s per GB300 (fwd+constrain+verify)"


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def algorithmic_bytes(shape, batch, L, ctx_len):
    """Bytes one block must move at minimum: drafter layer weights, LM-head rows, context K/V reads."""
    s = shape
    layer = (s.qkv_rows * s.d_model + s.d_model * s.n_q_heads * s.head_dim + 2 * s.d_ff * s.d_model
             + s.d_model * s.d_ff) * 2
    lm = s.vocab * s.d_model * 2
    kv = int(np.sum(ctx_len)) * s.n_layers * 2 * s.n_kv_heads * s.head_dim * 2
    return s.n_layers * layer, lm, kv


class ClockSampler:
    def __init__(self, out_path):
        self.out_path = out_path
        self.proc = None

    def __enter__(self):
        try:
            self.f = open(self.out_path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                 "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self, gpu_index=0):
        try:
            rows = [ln.split(",") for ln in open(self.out_path) if ln.strip()]
        except Exception:
            rows = []
        rows = [[c.strip() for c in r] for r in rows if len(r) >= 9 and r[0].strip() == str(gpu_index)]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def max_over_ranks(elapsed_ms, world, device):
    """The timed region's length as the slowest rank saw it (all ranks get the same number)."""
    if world == 1:
        return float(elapsed_ms)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(elapsed_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world, tokens_per_step, steps, elapsed_ms):
    """Whole-job draft tokens/s: every replica drafts `tokens_per_step` per step; time = slowest rank."""
    return world * tokens_per_step * steps / (elapsed_ms / 1e3)


def run_oracle_block(om, wl, kv, target, layout):
    import oracle
    t0 = time.perf_counter()
    hid = oracle.draft_block(om, kv, wl.t_cap, wl.ctx_len, wl.anchor, wl.mask_id, wl.block_len)
    toks, _, _ = oracle.constrain_argmax(om, hid, wl.batch, wl.block_len, layout=layout)
    if layout is None:
        oracle.verify(0, toks, target)
    else:
        oracle.verify(1, toks, layout=layout, rule=layout["rule"], pad_id=layout["pad_id"])
    return time.perf_counter() - t0


def oracle_sample(wl, w, kv_np, target):
    """The oracle as it stands on one block of request 0 (a bounded sample of the workload)."""
    import dataclasses
    import oracle
    om = oracle.Model(wl.shape, w)
    one = dataclasses.replace(wl, batch=1, ctx_len=wl.ctx_len[:1], anchor=wl.anchor[:1], t_cap=int(wl.ctx_len[0]))
    kv1 = np.ascontiguousarray(kv_np[:, :1, :, :, :one.t_cap])
    lay = wl.layout
    return om, one, kv1, (target[:1] if target is not None else None), lay


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="text_4b_b1")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()

    import torch
    import synth

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local_rank)
        dist.init_process_group(backend)

    wl = synth.make_workload(args.workload)
    s = wl.shape
    L, B = wl.block_len, wl.batch
    draft_tokens_per_step = B * (L - 1)
    config = {"workload": args.workload, "batch": B, "block_len": L, "context": wl.ctx_len.tolist() if B <= 4 else
              [int(wl.ctx_len.min()), int(wl.ctx_len.max())], "d_model": s.d_model, "layers": s.n_layers,
              "vocab": s.vocab, "layout": "unconstrained" if wl.layout is None else args.workload.split("_")[1],
              "l2": "inputs larger than L2 (1.83 GB weights streamed per step)"}

    if args.impl == "reference":
        # the CPU oracle, as it stands, on the host cores: rank 0 only
        if rank != 0:
            return
        import oracle
        oracle.build()
        w = synth.make_weights(s, wl.seed)
        kv = synth.make_kv_store(s, B, wl.t_cap, wl.seed + 5)
        om, one, kv1, _, lay = oracle_sample(wl, w, kv, None)
        target = None
        if lay is None:
            rng = np.random.default_rng(wl.seed + 9)
            target = rng.integers(0, s.vocab, (1, L)).astype(np.int32)
        for _ in range(max(0, min(args.warmup, 1))):
            run_oracle_block(om, one, kv1, target, lay)
        times = [run_oracle_block(om, one, kv1, target, lay) for _ in range(args.steps)]
        t = float(np.sum(times))
        v = args.steps * (L - 1) / t
        cores = oracle.num_threads()
        line = {"metric": METRIC, "value": v, "unit": "draft tokens/s", "n_gpus": args.gpus, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config,
                "impl": "reference",
                "cpu_baseline": {"value": v, "unit": "draft tokens/s", "cores": cores, "kind": "oracle",
                                 "sample": "one block of request 0 per step (draft + constrained argmax + verify)"},
                "e2e": {"value": v, "unit": "draft tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    import block_diffusion_speculative_non_gb300 as pkg
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    hbm_peak, tc_peak, peak_kind = peaks()

    w = synth.make_weights(s, wl.seed)
    dr = pkg.Drafter(s, w, B, L, wl.t_cap, device=dev)
    feats = synth.make_features(s, int(wl.row_off[-1]), wl.seed + 1)
    stream = torch.cuda.current_stream(dev)
    # context preparation (timed separately, once)
    fd, row_off_d, _ = dr.prepare_context(B, wl.row_off, feats)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    pkg.fpd_prepare_context(dr.handle, B, int(wl.row_off[-1]), row_off_d, None, fd, dr.kv_store, dr.t_cap,
                            dr.workspace, dr.ws_bytes, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    prepare_ms = e0.elapsed_time(e1)

    ctx_len = torch.from_numpy(wl.ctx_len).to(dev)
    anchor = torch.from_numpy(wl.anchor).to(dev)
    hidden = torch.empty(B * L, s.d_model, dtype=torch.bfloat16, device=dev)
    tokens = torch.empty(B, L - 1, dtype=torch.int32, device=dev)
    accept = torch.empty(B, dtype=torch.int32, device=dev)
    committed = torch.empty(B, L, dtype=torch.int32, device=dev)
    valid = torch.empty(B, dtype=torch.int32, device=dev)
    lay_d = rule_d = None
    if wl.layout is not None:
        lay_d, rule_d = pkg.Drafter.layout(wl.layout, B, L, dev)
    # target rows: Geometric(p) agreement with the drafter's own ids (text mode)
    pkg.fpd_draft_block(dr.handle, B, L, dr.kv_store, dr.t_cap, ctx_len, anchor, wl.mask_id, hidden, None,
                        dr.workspace, dr.ws_bytes, stream)
    pkg.fpd_constrain_argmax(dr.handle, B, L, hidden, lay_d, tokens, None, dr.workspace, dr.ws_bytes, stream)
    torch.cuda.synchronize()
    target_np = None
    if wl.layout is None:
        target_np, _ = synth.make_target_rows(tokens.cpu().numpy(), s.vocab, wl.geo_p or 0.25, wl.seed + 2)
    target = torch.from_numpy(target_np).to(dev) if target_np is not None else None

    def do_draft(st):
        pkg.fpd_draft_block(dr.handle, B, L, dr.kv_store, dr.t_cap, ctx_len, anchor, wl.mask_id, hidden, None,
                            dr.workspace, dr.ws_bytes, st)

    def do_argmax(st):
        pkg.fpd_constrain_argmax(dr.handle, B, L, hidden, lay_d, tokens, None, dr.workspace, dr.ws_bytes, st)

    def do_verify(st):
        if wl.layout is None:
            pkg.fpd_verify(0, B, L, tokens, target, None, None, -1, accept, committed, valid, st)
        else:
            pkg.fpd_verify(1, B, L, tokens, None, lay_d, rule_d, wl.layout["pad_id"], accept, committed, valid, st)

    # eager warm-up (also counts the kernels one step launches)
    for _ in range(max(3, args.warmup)):
        n0 = pkg.fpd_kernel_launches()
        do_draft(stream)
        do_argmax(stream)
        do_verify(stream)
        launches_per_step = pkg.fpd_kernel_launches() - n0
    torch.cuda.synchronize()

    # the step as three CUDA graphs (draft | LM head + argmax | verify) so the LM-head call can be timed live
    cap = torch.cuda.Stream(dev)
    graphs = []
    for fn in (do_draft, do_argmax, do_verify):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            fn(torch.cuda.current_stream(dev))
        graphs.append(g)
    g_draft, g_argmax, g_verify = graphs
    ev_lm = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]

    def step(i=None):
        g_draft.replay()
        if i is not None:
            ev_lm[i][0].record(stream)
        g_argmax.replay()
        if i is not None:
            ev_lm[i][1].record(stream)
        g_verify.replay()

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    t0e, t1e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clock_fd, clock_path = tempfile.mkstemp(prefix=f"fpd_bench_clocks_r{rank}_", suffix=".csv")
    os.close(clock_fd)
    with ClockSampler(clock_path) as cs:
        barrier()
        torch.cuda.synchronize()
        t0e.record(stream)
        for i in range(args.steps):
            step(i)
        t1e.record(stream)
        torch.cuda.synchronize()
        barrier()
    launches = launches_per_step * args.steps      # graph replays: the kernels of one step, K times
    elapsed_ms = t0e.elapsed_time(t1e)
    lm_ms = float(np.mean([a.elapsed_time(b) for a, b in ev_lm]))
    assert pkg.fpd_device_status(stream) == 0, "device-side check failed"
    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)
    ms_per_step = elapsed_ms / args.steps
    value = replica_throughput(world, draft_tokens_per_step, args.steps, elapsed_ms)

    # ---- end to end through the C ABI with host buffers: H2D of the step's inputs, D2H of its results --------
    a_h = torch.from_numpy(wl.anchor.copy()).pin_memory()
    t_h = torch.from_numpy(target_np.copy()).pin_memory() if target_np is not None else None
    acc_h = torch.empty(B, dtype=torch.int32).pin_memory()
    com_h = torch.empty(B, L, dtype=torch.int32).pin_memory()
    h2d = a_h.numel() * 4 + (t_h.numel() * 4 if t_h is not None else 0)
    d2h = acc_h.numel() * 4 + com_h.numel() * 4
    e2e_steps = max(10, args.steps // 2)
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        anchor.copy_(a_h, non_blocking=True)
        if t_h is not None:
            target.copy_(t_h, non_blocking=True)
        step()
        acc_h.copy_(accept, non_blocking=True)
        com_h.copy_(committed, non_blocking=True)
        stream.synchronize()
    e2e_s = time.perf_counter() - t0
    e2e_value = world * draft_tokens_per_step * e2e_steps / e2e_s

    # ---- roofline of the dominant kernel (LM head call: final norm + LM-head GEMM/argmax + decode) -------
    layer_b, lm_b, kv_b = algorithmic_bytes(s, B, L, wl.ctx_len)
    lm_bytes = lm_b + B * (L - 1) * s.d_model * 2
    achieved = lm_bytes / (lm_ms * 1e-3) / 1e9
    block_bytes = layer_b + lm_b + kv_b
    roofline = {"bound": "hbm", "kernel": "fpd_constrain_argmax (LM head, 128-id x token tiles, tcgen05)",
                "achieved": achieved, "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
                "peak_kind": f"{peak_kind} (copy, burst)", "traffic": None,
                "block_bytes": block_bytes, "block_frac": block_bytes / (ms_per_step * 1e-3) / 1e9 / hbm_peak}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        try:
            import oracle
            oracle.build()
            # the oracle's inputs come from the seeded generators only (timing sample, values irrelevant)
            kv_np = synth.make_kv_store(s, 1, int(wl.ctx_len[0]), wl.seed + 5)
            tgt_np = np.random.default_rng(wl.seed + 9).integers(0, s.vocab, (1, L)).astype(np.int32)
            om, one, kv1, tgt1, lay = oracle_sample(wl, w, kv_np, tgt_np)
            dt = run_oracle_block(om, one, kv1, tgt1, lay)
            cpu = {"value": (L - 1) / dt, "unit": "draft tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
                   "sample": "one block of request 0 (draft + constrained argmax + verify), fp64 oracle"}
        except Exception as e:  # the baseline is reported, never required
            cpu = {"value": None, "unit": "draft tokens/s", "cores": None, "kind": "oracle", "sample": f"failed: {e}"}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "draft tokens/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": config,
                "blocks_per_s": world * B * args.steps / (elapsed_ms / 1e3), "prepare_ms": prepare_ms,
                "roofline": roofline, "cpu_baseline": cpu,
                "e2e": {"value": e2e_value, "unit": "draft tokens/s", "h2d_bytes_per_step": h2d,
                        "d2h_bytes_per_step": d2h},
                "gpu_launches": int(launches), "clocks": cs.summary(local_rank)}
        print(json.dumps(line), flush=True)
    try:
        os.remove(clock_path)
    except OSError:
        pass
    dr.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
